"""Host-side pieces of bench.py on CPU: the algorithmic byte count (each pool
slot read once, shared blocks once) and the oracle baseline's thread-count
self-check."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from oracle.allocator import ReferenceAllocator  # noqa: E402
from workloads import CONFIGS, build_tables, make_case  # noqa: E402


def test_unique_tokens_counts_shared_blocks_once():
    # sequences 0 and 1 share block 7 (full); 0 holds 20 tokens, 1 holds 17
    tables = np.array([[7, 3], [7, 9]], np.int32)
    assert bench.unique_tokens(tables, np.array([20, 17])) == 16 + 4 + 1
    # a block shared with different fill: the longer prefix counts
    tables = np.array([[5], [5]], np.int32)
    assert bench.unique_tokens(tables, np.array([3, 11])) == 11
    assert bench.unique_tokens(tables, np.array([0, 0])) == 0


def test_step_bytes_of_the_shared_prefix_workload():
    cfg = CONFIGS[4]
    case = make_case(cfg)
    tables, _, _, lens = build_tables(case, ReferenceAllocator(case.num_blocks, 16, case.free_order))
    b = bench.step_bytes(cfg, lens, tables)
    per_tok = cfg.n_kv_heads * 128 * 2 * 2
    children = sum(1 for i in cfg.shared_children if i < len(lens))
    assert b["kv_logical"] == int(lens.sum()) * per_tok
    assert b["kv"] == (int(lens.sum()) - (children - 1) * cfg.shared_prefix) * per_tok
    assert b["total"] == b["kv"] + b["new_rows"] + b["q"] + b["out"] + b["tables"]
    # no sharing: the two counts agree
    tiny = CONFIGS[1]
    case = make_case(tiny)
    tables, _, _, lens = build_tables(case, ReferenceAllocator(case.num_blocks, 16, case.free_order))
    b = bench.step_bytes(tiny, lens, tables)
    assert b["kv"] == b["kv_logical"]


def test_oracle_result_does_not_depend_on_threads():
    cfg = CONFIGS[1]
    case = make_case(cfg)
    tables, _, _, lens = build_tables(case, ReferenceAllocator(case.num_blocks, 16, case.free_order))
    many = bench.OracleSample(cfg, case, tables, lens, 4)
    one = bench.OracleSample(cfg, case, tables, lens, 1)
    assert bench.thread_count_diff(many, one, many.groups) == 0.0


def test_both_arms_describe_the_workload_identically():
    cfg = CONFIGS[3]
    case = make_case(cfg)
    tables, _, _, lens = build_tables(case, ReferenceAllocator(case.num_blocks, 16, case.free_order))
    a = bench.config_dict(cfg, case, lens, tables, 0, bench.GB300_L2_BYTES)
    case2 = make_case(cfg)
    tables2, _, _, lens2 = build_tables(case2, ReferenceAllocator(case2.num_blocks, 16, case2.free_order))
    b = bench.config_dict(cfg, case2, lens2, tables2, 0, bench.GB300_L2_BYTES)
    assert a == b
    assert a["workload"] == cfg.name and a["tokens_attended"] == int(lens.sum())


def test_parity_record_bar_and_native_check():
    rng = np.random.default_rng(0)
    ref = rng.standard_normal((4, 8, 128))
    ok = bench.parity_record(ref + 1e-4, ref)
    assert ok["pass"] and abs(ok["max_abs_err"] - 1e-4) < 1e-9
    bad = bench.parity_record(ref + 3e-3, ref)
    assert not bad["pass"]
    nan = ref.copy()
    nan[0, 0, 0] = np.nan
    assert not bench.parity_record(nan, ref)["pass"]
    import torch
    rn = torch.from_numpy(ref).float().to(torch.bfloat16).double().numpy()
    rec = bench.parity_record(ref, ref, got_native=rn, dtype=torch.bfloat16, v_absmax=4.0)
    assert rec["native_16bit"]["beyond_one_ulp"] == 0
    off = rn * (1 + 2.0 ** -5)  # four bf16 ulps off
    rec = bench.parity_record(ref, ref, got_native=off, dtype=torch.bfloat16, v_absmax=4.0)
    assert rec["native_16bit"]["beyond_one_ulp"] > 0
