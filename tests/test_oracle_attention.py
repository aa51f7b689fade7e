"""Pins for the fp64 paged-decode oracle, each against something other than the
oracle itself: IEEE decoders of numpy/torch, torch's fp64 scaled-dot-product
attention on the un-paged cache, closed forms, invariants and brute force.

The decode definition is that of "Serving", section 23.4 Paged Attention
(blocks plus a per-sequence table) over an exact cache ("The KV Cache" teaser
on the inference-serving tag page: cached and recomputed results match)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests._util import BS, bits, dtype_code, pool_from_dense, to_bits

DTYPES = [torch.float16, torch.bfloat16]


def test_fp16_decoder_all_patterns():
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_bits_to_double(p) for p in pats.tolist()])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_bf16_decoder_all_patterns():
    pats = np.arange(1 << 16, dtype=np.int32).astype(np.int16)
    ref = torch.from_numpy(pats).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_bits_to_double(p) for p in pats.view(np.uint16).tolist()])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def _random_paged(seed, lens, Hq, Hkv, d, dt, extra_blocks=5, fill=0.0):
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    q = torch.randn(B, Hq, d, generator=g).to(dt)
    dense_k = [torch.randn(Hkv, L, d, generator=g).to(dt) for L in lens]
    dense_v = [torch.randn(Hkv, L, d, generator=g).to(dt) for L in lens]
    nbs = [max(1, -(-L // BS)) for L in lens]
    N = sum(nbs) + extra_blocks
    perm = torch.randperm(N, generator=g).numpy()
    kp, tables = pool_from_dense([x.double().numpy() for x in dense_k], nbs, N, perm, fill=fill)
    vp, _ = pool_from_dense([x.double().numpy() for x in dense_v], nbs, N, perm, fill=fill)
    kt, kb = to_bits(kp, dt)
    vt, vb = to_bits(vp, dt)
    return dict(q=q, dense_k=dense_k, dense_v=dense_v, kp=kb, vp=vb, tables=tables,
                lens=np.array(lens, np.int32), N=N, perm=perm)


def _sdpa_dense(q, dense_k, dense_v, scale, i):
    """torch fp64 SDPA (grouped-query mapping by the library) on sequence i."""
    qi = q[i].double()[None, :, None, :]                  # [1][Hq][1][d]
    ki = dense_k[i].double()[None]                        # [1][Hkv][L][d]
    vi = dense_v[i].double()[None]
    o = F.scaled_dot_product_attention(qi, ki, vi, scale=scale, enable_gqa=True)
    return o[0, :, 0, :].numpy()


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("Hq,Hkv", [(12, 2), (32, 8), (4, 4)])
def test_matches_torch_sdpa_on_unpaged_cache(dt, Hq, Hkv):
    lens = [1, 15, 16, 17, 100, 257]
    c = _random_paged(7 + Hq, lens, Hq, Hkv, 128, dt)
    scale = 1 / math.sqrt(128)
    got = oracle.paged_decode(bits(c["q"]), c["kp"], c["vp"], dtype_code(dt), c["tables"], c["lens"], scale)
    for i in range(len(lens)):
        ref = _sdpa_dense(c["q"], c["dense_k"], c["dense_v"], scale, i)
        np.testing.assert_allclose(got[i], ref, rtol=0, atol=1e-12)


def test_unused_slots_are_never_read():
    """NaN in every slot outside the sequences (tails, spare blocks) must not
    reach the output."""
    lens = [3, 17, 31]
    c = _random_paged(11, lens, 8, 2, 128, torch.float16, fill=np.nan)
    got = oracle.paged_decode(bits(c["q"]), c["kp"], c["vp"], 0, c["tables"], c["lens"], 0.1)
    assert np.isfinite(got).all()


def test_block_permutation_invariance_bit_exact():
    lens = [40, 70, 5]
    c = _random_paged(3, lens, 12, 2, 128, torch.bfloat16)
    base = oracle.paged_decode(bits(c["q"]), c["kp"], c["vp"], 1, c["tables"], c["lens"], 0.08)
    rng = np.random.default_rng(0)
    pi = rng.permutation(c["N"])
    kp2 = np.empty_like(c["kp"]); vp2 = np.empty_like(c["vp"])
    kp2[pi] = c["kp"]; vp2[pi] = c["vp"]
    t2 = np.where(c["tables"] >= 0, pi[np.maximum(c["tables"], 0)], -1).astype(np.int32)
    got = oracle.paged_decode(bits(c["q"]), kp2, vp2, 1, t2, c["lens"], 0.08)
    assert np.array_equal(base, got)


def test_shared_prefix_equals_unshared_copy():
    """Two sequences whose first 32 tokens live in the same physical blocks
    give the same result as when each has its own copy."""
    g = torch.Generator().manual_seed(5)
    Hkv, Hq, d = 2, 4, 128
    kp = torch.randn(10, Hkv, BS, d, generator=g).half()
    vp = torch.randn(10, Hkv, BS, d, generator=g).half()
    kp[5:7] = kp[0:2]; vp[5:7] = vp[0:2]          # blocks 5,6 copy blocks 0,1
    q = torch.randn(2, Hq, d, generator=g).half()
    lens = np.array([40, 45], np.int32)
    shared = np.array([[0, 1, 2], [0, 1, 3]], np.int32)
    copied = np.array([[0, 1, 2], [5, 6, 3]], np.int32)
    a = oracle.paged_decode(bits(q), bits(kp), bits(vp), 0, shared, lens, 0.1)
    b = oracle.paged_decode(bits(q), bits(kp), bits(vp), 0, copied, lens, 0.1)
    assert np.array_equal(a, b)


def _single(q_vec, K_rows, V_rows, scale, dt=torch.float16, d=128):
    """One sequence, one head, the given rows in one or more blocks."""
    L = K_rows.shape[0]
    nb = -(-L // BS)
    kp = np.zeros((nb, 1, BS, d)); vp = np.zeros((nb, 1, BS, d))
    kp.reshape(nb * BS, d)[:L] = K_rows
    vp.reshape(nb * BS, d)[:L] = V_rows
    tables = np.arange(nb, dtype=np.int32)[None]
    _, qb = to_bits(np.asarray(q_vec)[None, None, :], dt)
    _, kb = to_bits(kp, dt)
    _, vb = to_bits(vp, dt)
    return oracle.paged_decode(qb, kb, vb, dtype_code(dt), tables, np.array([L], np.int32), scale)[0, 0]


def test_closed_form_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    v = np.round(rng.standard_normal(128) * 64) / 64
    out = _single(rng.standard_normal(128), rng.standard_normal((1, 128)), v[None], 0.3)
    assert np.array_equal(out, v)


def test_closed_form_zero_query_is_mean_of_values():
    rng = np.random.default_rng(2)
    L = 37
    V = np.round(rng.standard_normal((L, 128)) * 8) / 8
    out = _single(np.zeros(128), rng.standard_normal((L, 128)), V, 0.5)
    np.testing.assert_allclose(out, V.mean(axis=0), rtol=0, atol=1e-14)


def test_closed_form_zero_scale_is_mean_of_values():
    rng = np.random.default_rng(3)
    L = 20
    V = np.round(rng.standard_normal((L, 128)) * 8) / 8
    out = _single(rng.standard_normal(128), rng.standard_normal((L, 128)), V, 0.0)
    np.testing.assert_allclose(out, V.mean(axis=0), rtol=0, atol=1e-14)


def test_closed_form_two_tokens_weights_three_to_one():
    """Logits ln3 and 0 give weights 3/4 and 1/4 - pins the sign of the
    scale, the exponent and the normalisation."""
    q = np.zeros(128); q[0] = 1.0
    K = np.zeros((2, 128)); K[0, 0] = 1.0
    V = np.zeros((2, 128)); V[0, 0] = 1.0; V[1, 1] = 1.0
    out = _single(q, K, V, math.log(3.0))
    expect = np.zeros(128); expect[0] = 0.75; expect[1] = 0.25
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-15)


def test_closed_form_dominant_logit_selects_its_row():
    L = 33
    q = np.zeros(128); q[5] = 8.0
    K = np.zeros((L, 128)); K[29, 5] = 8.0           # logit 64*scale only at t=29
    rng = np.random.default_rng(4)
    V = np.round(rng.standard_normal((L, 128)) * 4) / 4
    out = _single(q, K, V, 16.0)                     # 1024 above the rest
    np.testing.assert_allclose(out, V[29], rtol=0, atol=1e-300)


def test_grouped_query_mapping_closed_form():
    """V of kv head g is the constant g+1, so out[i][h] reveals which kv head
    query head h used: h // (Hq/Hkv)."""
    Hq, Hkv, d = 12, 3, 128
    G = Hq // Hkv
    rng = np.random.default_rng(6)
    kp = rng.standard_normal((4, Hkv, BS, d))
    vp = np.zeros((4, Hkv, BS, d))
    for g in range(Hkv):
        vp[:, g] = g + 1
    _, kb = to_bits(kp, torch.float16); _, vb = to_bits(vp, torch.float16)
    _, qb = to_bits(rng.standard_normal((1, Hq, d)), torch.float16)
    out = oracle.paged_decode(qb, kb, vb, 0, np.array([[2, 0, 3]], np.int32), np.array([40], np.int32), 0.1)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], h // G + 1, rtol=0, atol=1e-13)


def test_brute_force_tiny():
    """Pure-Python loops straight from the definition (no max subtraction),
    block size 4 and width 8, against the oracle."""
    bs, d, Hq, Hkv = 4, 8, 4, 2
    rng = np.random.default_rng(9)
    lens = [5, 9, 1]
    N = 9
    kp = np.round(rng.standard_normal((N, Hkv, bs, d)) * 16) / 16
    vp = np.round(rng.standard_normal((N, Hkv, bs, d)) * 16) / 16
    qv = np.round(rng.standard_normal((3, Hq, d)) * 16) / 16
    tables = np.array([[4, 1, -1], [0, 8, 6], [3, -1, -1]], np.int32)
    scale = 0.37
    _, kb = to_bits(kp, torch.float16); _, vb = to_bits(vp, torch.float16)
    _, qb = to_bits(qv, torch.float16)
    got = oracle.paged_decode(qb, kb, vb, 0, tables, np.array(lens, np.int32), scale)
    for i, L in enumerate(lens):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            ws, rows = [], []
            for t in range(L):
                blk = int(tables[i][t // bs])
                krow = kp[blk][g][t % bs]
                s = scale * sum(float(qv[i][h][k]) * float(krow[k]) for k in range(d))
                ws.append(math.exp(s))
                rows.append(vp[blk][g][t % bs])
            z = sum(ws)
            ref = [sum(w * float(r[k]) for w, r in zip(ws, rows)) / z for k in range(d)]
            np.testing.assert_allclose(got[i][h], ref, rtol=0, atol=1e-12)


def test_zero_length_gives_zero_row_and_sampled_rows_match_full():
    c = _random_paged(12, [0, 33, 64], 8, 4, 128, torch.bfloat16)
    full = oracle.paged_decode(bits(c["q"]), c["kp"], c["vp"], 1, c["tables"], c["lens"], 0.09)
    assert not full[0].any()
    rows = [3, 9, 23, 17]
    part = oracle.paged_decode(bits(c["q"]), c["kp"], c["vp"], 1, c["tables"], c["lens"], 0.09, rows=rows)
    flat = full.reshape(-1, 128)
    assert np.array_equal(part, flat[rows])


def test_out_of_range_block_is_refused():
    c = _random_paged(13, [20], 4, 2, 128, torch.float16)
    bad = c["tables"].copy(); bad[0, 1] = c["N"]
    with pytest.raises(ValueError):
        oracle.paged_decode(bits(c["q"]), c["kp"], c["vp"], 0, bad, c["lens"], 0.1)


def test_threads_do_not_change_the_result():
    c = _random_paged(14, [100, 31, 200, 64], 12, 2, 128, torch.bfloat16)
    a = oracle.paged_decode(bits(c["q"]), c["kp"], c["vp"], 1, c["tables"], c["lens"], 0.08, threads=1)
    b = oracle.paged_decode(bits(c["q"]), c["kp"], c["vp"], 1, c["tables"], c["lens"], 0.08, threads=4)
    assert np.array_equal(a, b)
