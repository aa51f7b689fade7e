"""Several new query tokens per sequence (pa_decode_multi) against the fp64
oracle: causal within the new tokens, GQA and MHA layouts, fp16 and bf16,
ragged new-token counts including a whole fresh sequence and sequences with
none, native 16-bit output, and the error path."""
import numpy as np
import pytest
import torch

from oracle.multi_query import paged_multi_query

from ._gpu import GpuCase, assert_close, assert_within_one_ulp16, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_227_gb300 as pa
    return pa


def run_multi(pa, c, news, out_dtype=torch.float32, seed=0):
    news = np.asarray(news, dtype=np.int32)
    q_start = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    n_q = int(q_start[-1])
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(n_q, c.cfg.n_q_heads, 128, generator=g).to(c.dtype)
    pool = c.pool()
    out = torch.full((n_q, c.cfg.n_q_heads, 128), float("nan"), dtype=out_dtype, device="cuda")
    pa.pa_decode_multi(pool, q.cuda(), torch.from_numpy(q_start).cuda(), c.tables_dev(), c.lens_dev(),
                       c.case.scale, out)
    torch.cuda.synchronize()
    code, detail = pa.pa_check(pool)
    ref = paged_multi_query(bits(q), c.kp, c.vp, c.code, c.tables, c.dec_lens, q_start, c.case.scale)
    return out, ref, code, q


@pytest.mark.parametrize("cfg,news", [
    (1, [18, 1, 3, 32]),          # Qwen2.5-1.5B layout (G = 6, FMA values), fp16; sequence 0 wholly new
    (3, None),                    # LLaMA-3-8B layout (G = 4, tensor-core values), bf16
    (4, None),                    # Llama-2-13B MHA (G = 1), fp16
])
def test_matches_oracle(pa, cfg, news):
    lens = {1: None, 3: [40, 7, 130, 16, 1, 65], 4: [2100, 2500, 2048, 3000, 2200, 2600]}[cfg]
    c = GpuCase(cfg, lens=lens) if lens else GpuCase(cfg)
    if news is None:
        rnd = np.random.default_rng(cfg)
        news = [int(rnd.integers(0, min(L, 24) + 1)) for L in c.dec_lens]
        news[1] = 0                 # a sequence with no new tokens
        if cfg == 3:
            news[0] = int(c.dec_lens[0])  # the whole sequence is new
    out, ref, code, _ = run_multi(pa, c, news)
    assert code == 0
    assert_close(out, ref, f"multi cfg{cfg}")


@pytest.mark.parametrize("news", [
    [2] * 6,                      # 8 columns a sequence: one 8-column segment each
    [3] * 6,                      # more than 8 on average: 16 columns, 4 empty
    [5, 9, 1, 4, 16, 0],          # 16 columns; packs of 4 tokens and a partial last pack
])
def test_packing_widths(pa, news):
    """Tokens packed 8 or 16 columns to a segment (chosen from the average
    new-token count), with empty columns and partial last packs."""
    c = GpuCase(3, lens=[40, 70, 130, 16, 300, 65])
    out, ref, code, _ = run_multi(pa, c, news)
    assert code == 0
    assert_close(out, ref, f"multi packing {news}")


def test_one_new_token_is_bit_identical_to_split_decode(pa):
    """With one new token per sequence the rows are the sequences themselves:
    same lengths, same tables, same balanced split, same bits."""
    c = GpuCase(3, lens=[33, 700, 5, 1200, 64, 250])
    out, ref, code, q = run_multi(pa, c, [1] * 6)
    assert code == 0
    assert_close(out, ref, "multi with one token")
    dec = torch.empty_like(out)
    pa.pa_decode_split(c.pool(), q.cuda(), c.tables_dev(), c.lens_dev(), c.case.scale, dec)
    torch.cuda.synchronize()
    assert torch.equal(out, dec)


def test_native_16bit_output_within_one_ulp(pa):
    c = GpuCase(3, lens=[100, 17, 48])
    out, ref, code, _ = run_multi(pa, c, [5, 17, 2], out_dtype=torch.bfloat16)
    assert code == 0
    assert_within_one_ulp16(out.cpu(), ref, torch.bfloat16, "multi bf16 out", vmax=c.vmax())


def test_speculative_verification_shape_full_size(pa):
    """The LLaMA-3-8B batch-64 workload with 4 drafted tokens per sequence."""
    c = GpuCase(3)
    out, ref, code, _ = run_multi(pa, c, [4] * len(c.dec_lens))
    assert code == 0
    assert_close(out, ref, "multi 4 tokens, batch 64")


def test_more_new_tokens_than_the_sequence_is_reported(pa):
    c = GpuCase(3, lens=[10, 20])              # the sequences hold 11 and 21 tokens
    news = np.array([3, 25], np.int32)         # 25 > 21
    q_start = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    pool = c.pool()
    q = torch.randn(int(q_start[-1]), c.cfg.n_q_heads, 128).to(c.dtype).cuda()
    out = torch.full((q.shape[0], c.cfg.n_q_heads, 128), 7.0, device="cuda")
    pa.pa_decode_multi(pool, q, torch.from_numpy(q_start).cuda(), c.tables_dev(), c.lens_dev(), c.case.scale, out)
    torch.cuda.synchronize()
    code, _ = pa.pa_check(pool)
    assert code == pa.PA_ERR_DEVICE_CHECK
    assert (out[3:7] == 0).all(), "rows that would sit before position 0 output zeros"
    assert torch.isfinite(out[7:]).all() and not (out[7:] == 7.0).any()


@pytest.mark.parametrize("q_start", [
    [0, 3, 2, 6],                 # decreases
    [1, 3, 4, 6],                 # does not start at 0
    [0, 2, 4, 5],                 # ends before n_q = 6
])
def test_malformed_q_start_is_reported(pa, q_start):
    """Only rows inside [0, n_q) are ever touched; the plan reports the
    malformed offsets through pa_check."""
    c = GpuCase(3, lens=[10, 20, 30])
    pool = c.pool()
    n_q = 6
    q = torch.randn(n_q, c.cfg.n_q_heads, 128).to(c.dtype).cuda()
    out = torch.zeros((n_q, c.cfg.n_q_heads, 128), device="cuda")
    qs = torch.tensor(q_start, dtype=torch.int32, device="cuda")
    pa.pa_decode_multi(pool, q, qs, c.tables_dev(), c.lens_dev(), c.case.scale, out)
    torch.cuda.synchronize()
    code, _ = pa.pa_check(pool)
    assert code == pa.PA_ERR_DEVICE_CHECK
    assert torch.isfinite(out).all()
