"""Benchmark of one paged decode step on GB300.

A step is the whole hot path for one batch: the new token of every sequence
is written to its slot and attended together with the cached tokens (fused
append + balanced split-KV decode + log-sum-exp merge, pa_append_decode).
Default workload: LLaMA-3-8B layout (32 q / 8 kv heads, d 128, bf16), batch 64,
lognormal lengths (median 600, sigma 0.8, clipped to [16, 8192]), 16-token
blocks at random places in a pool 1.25x the needed size.

Output: one JSON line (rank 0).  `value` is algorithmic bytes per step (K/V
of every attended token, the new rows written, q, output, tables, lengths)
over the device time of the step, summed over ranks, in GB/s.  Inputs are
resident in HBM; L2 is flushed (a 2x-L2 buffer is read) before every timed
step.  `e2e` repeats the measurement through the same public calls with the
step's inputs copied from pinned host memory (one staging buffer, one copy)
and the output copied back inside the timed region.

`other_configs` carries the same measurement for the other workloads (the
tiny and batch-32 Qwen2.5-1.5B layouts, the Llama-2-13B shared-prefix
workload with its cascade, the long-context workload with the balanced split
and with fixed partitions), and `parity` the comparison of the timed step's
result (one extra call with fp32 output, same inputs and launch) with the fp64
oracle on the whole workload.

`--gpus N` without a launcher starts N ranks itself (one process per GPU,
weak scaling: every rank decodes its own batch; NCCL only for the barrier and
the max/sum over ranks).  Under a launcher, WORLD_SIZE must equal N.

`--impl reference` times the fp64 CPU oracle instead (the only other arm this
repository has), on a bounded sample of the same workload.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: KV GB/s vs GB300 HBM peak; µs per decode step"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=3, help="config number (default: the batch-64 LLaMA-3-8B layout)")
    ap.add_argument("--partition-blocks", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--row", default="decode",
                    choices=["decode", "multi-query", "cascade", "prefix-cache", "utilisation"],
                    help="decode: the headline step; the others time the further rows (one JSON line each)")
    ap.add_argument("--new-tokens", type=int, default=4, help="multi-query: new tokens per sequence")
    ap.add_argument("--no-other-configs", action="store_true", help="headline workload only")
    ap.add_argument("--clock-window", type=float, default=0.3,
                    help="seconds of untimed steps right after the timed ones, to sample clocks under load")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def unique_tokens(tables, dec_lens):
    """Pool token slots the step reads at least once: a sequence reads a prefix
    of each of its blocks, so a block shared by several sequences counts the
    longest of their prefixes in it, once."""
    longest = {}
    for i, L in enumerate(np.asarray(dec_lens).tolist()):
        for j in range(-(-L // 16)):
            b = int(tables[i, j])
            longest[b] = max(longest.get(b, 0), min(16, L - 16 * j))
    return sum(longest.values())


def step_bytes(cfg, dec_lens, tables, out_bytes=2):
    """Algorithmic bytes of one fused append + decode step.  K/V bytes count
    each pool slot read once (blocks shared by several sequences once); the
    bytes of every sequence's own view are `kv_logical`."""
    B = len(dec_lens)
    Hq, Hkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.d_head
    kv = unique_tokens(tables, dec_lens) * Hkv * d * 2 * 2  # K and V of every slot read
    kv_logical = int(np.sum(dec_lens)) * Hkv * d * 2 * 2
    new_rows = B * Hkv * d * 2 * 2                       # the new K/V rows written to the pool
    q = B * Hq * d * 2
    out = B * Hq * d * out_bytes
    nb = int(np.sum(-(-dec_lens // 16)))
    table = 4 * nb + 4 * B
    return {"kv": kv, "new_rows": new_rows, "q": q, "out": out, "tables": table,
            "total": kv + new_rows + q + out + table, "kv_logical": kv_logical}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index, enabled=True):
        self.proc = None
        self.device_index = device_index
        if not enabled:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


def traffic_record(workload):
    """DRAM bytes per launch of the decode kernel from the committed ncu summary,
    or None when the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[str(workload)]
        src = os.path.join(ROOT, "paged_kv_cache_227_gb300", "csrc", "decode.cu")
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if rec.get("decode_cu_sha256") != digest:
            return None
        return rec
    except Exception:
        return None


def reduce_over_ranks(times_ms, nbytes, device):
    """Weak scaling across ranks: every rank decodes its own batch, so the job's
    time is the slowest rank's (max of each timing) and its bytes are the sum
    of the ranks' bytes.  Returns (times, total bytes)."""
    t = torch.tensor(times_ms, dtype=torch.float64, device=device)
    b = torch.tensor([float(nbytes)], dtype=torch.float64, device=device)
    if torch.distributed.is_initialized() and torch.distributed.get_world_size() > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.all_reduce(b, op=torch.distributed.ReduceOp.SUM)
    return t.tolist(), b.item()


def build_inputs(cfg_key, rank, device):
    import paged_kv_cache_227_gb300 as pa
    from workloads import CONFIGS, build_tables, make_case
    cfg = CONFIGS[cfg_key]
    case = make_case(cfg, seed=1000 + cfg.key + 7919 * rank)
    alloc = pa.BlockAllocator(case.num_blocks, 16, case.free_order)
    tables, slots, cows, dec_lens = build_tables(case, alloc)
    assert not cows, "the benchmark workloads append into fresh or private blocks"
    return pa, cfg, case, tables, slots, dec_lens


class Flush:
    """L2 flush by READING a 2x-L2 buffer: the cache is left holding clean
    lines, so the timed step pays no write-back of a flush's dirty lines."""

    def __init__(self, device):
        self.l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.buf = torch.ones(2 * self.l2 // 4, dtype=torch.float32, device=device)
        self.sink = torch.zeros(1, dtype=torch.float32, device=device)

    def __call__(self):
        self.sink.add_(self.buf.sum())


def device_inputs(pa, cfg, case, tables, dec_lens, device):
    pool = pa.Pool(case.num_blocks, cfg.n_kv_heads, cfg.torch_dtype)
    pool.k.copy_(case.k_pool.to(device))
    pool.v.copy_(case.v_pool.to(device))
    return dict(pool=pool, q=case.q.to(device), k_new=case.k_new.to(device), v_new=case.v_new.to(device),
                bt=torch.from_numpy(tables).to(device), sl=torch.from_numpy(dec_lens).to(device))


def fused_step_fn(pa, d, case, out, partition_blocks, ws):
    """The fused step with its ctypes arguments marshalled once."""
    import ctypes
    stream = torch.cuda.current_stream()
    fn = pa.lib.pa_append_decode
    argv = (d["pool"].handle, ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["k_new"].data_ptr()),
            ctypes.c_void_p(d["v_new"].data_ptr()), ctypes.c_void_p(d["bt"].data_ptr()), d["bt"].shape[1],
            ctypes.c_void_p(d["sl"].data_ptr()), d["q"].shape[0], d["q"].shape[1], float(case.scale),
            ctypes.c_void_p(out.data_ptr()), pa._DTYPE_CODE[out.dtype], partition_blocks,
            ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(stream.cuda_stream))

    def step():
        code = fn(*argv)
        if code != 0:
            raise pa.PagedAttentionError(code, "pa_append_decode")
    return step


def time_steps(step, flush, K, W, profile=None):
    """W untimed then K timed calls of `step`, L2 flushed before each; CUDA
    events around each call (and the library's own events around its
    launches when `profile` is the package).  Returns µs lists."""
    for _ in range(max(W, 3)):
        flush()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if profile is not None:
        profile.pa_profile_start(K)
    torch.cuda.synchronize()
    for k in range(K):
        flush()
        ev[k][0].record()
        step()
        ev[k][1].record()
    torch.cuda.synchronize()
    step_us = [a.elapsed_time(b) * 1e3 for a, b in ev]
    kern_us = [x * 1e3 for x in profile.pa_profile_stop(K)] if profile is not None else None
    return step_us, kern_us


def run_ours(args, rank, world, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    pa, cfg, case, tables, slots, dec_lens = build_inputs(args.workload, rank, device)
    d = device_inputs(pa, cfg, case, tables, dec_lens, device)
    pool, q = d["pool"], d["q"]
    out = torch.empty(q.shape, dtype=cfg.torch_dtype, device=device)
    ws = pa.workspace_for(pool, q, d["bt"], args.partition_blocks)
    nbytes = step_bytes(cfg, dec_lens, tables)
    flush = Flush(device)
    step = fused_step_fn(pa, d, case, out, args.partition_blocks, ws)
    launches_per_step = 3  # the append, the decode (its dependent) and the merge of split segments

    # clocks are sampled from before the warm-up to the end of an untimed
    # window of steps right after the timed ones (the timed region alone is
    # shorter than the sampling period)
    clocks = ClockSampler(local, enabled=(rank == 0 and not args.no_clocks))
    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    torch.cuda.synchronize()
    code, detail = pa.pa_check(pool)
    assert code == 0, (pa.strerror(code), detail)

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    pa.pa_profile_start(K)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for k in range(K):
        flush()
        ev[k][0].record()
        step()
        ev[k][1].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kern_ms = pa.pa_profile_stop(K)
    assert len(kern_ms) == K, "every timed step must record its decode kernel"
    t_win = time.perf_counter()
    while time.perf_counter() - t_win < args.clock_window:
        for _ in range(50):
            flush()
            step()
        torch.cuda.synchronize()
    clock_info = clocks.stop()
    mean_ms = float(np.mean(step_ms))
    kern_mean = float(np.mean(kern_ms))
    code, detail = pa.pa_check(pool)
    assert code == 0, (pa.strerror(code), detail)

    # end to end through the public call: the step's inputs live in one pinned
    # host staging buffer (q | k_new | v_new | tables | lengths, 256-byte
    # aligned parts), copied in with one copy; the output is copied out
    parts = [case.q, case.k_new, case.v_new, torch.from_numpy(tables), torch.from_numpy(dec_lens)]
    offs, n = [], 0
    for t in parts:
        offs.append(n)
        n += (t.numel() * t.element_size() + 255) // 256 * 256
    stage_h = torch.empty(n, dtype=torch.uint8).pin_memory()
    stage_d = torch.empty(n, dtype=torch.uint8, device=device)
    views_d = []
    for t, o in zip(parts, offs):
        nb = t.numel() * t.element_size()
        stage_h[o:o + nb].copy_(t.contiguous().view(-1).view(torch.uint8))
        views_d.append(stage_d[o:o + nb].view(t.dtype).view(t.shape))
    q_e, kn_e, vn_e, bt_e, sl_e = views_d
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in parts)
    d2h = out_h.numel() * out_h.element_size()
    KE = min(args.e2e_steps, K)
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(KE)]
    torch.cuda.synchronize()
    for k in range(KE):
        flush()
        eev[k][0].record()
        stage_d.copy_(stage_h, non_blocking=True)
        pa.pa_append_decode(pool, q_e, kn_e, vn_e, bt_e, sl_e, case.scale, out,
                            partition_blocks=args.partition_blocks, workspace=ws)
        out_h.copy_(out, non_blocking=True)
        eev[k][1].record()
    torch.cuda.synchronize()
    e2e_ms = float(np.mean([a.elapsed_time(b) for a, b in eev]))

    # the timed step's result: the last timed call's native output, and one
    # more call with the same inputs and launch whose output is fp32 (the
    # kernel's arithmetic before the final rounding), for the oracle leg
    out_native = out.float().cpu().numpy()
    out32 = torch.empty(q.shape, dtype=torch.float32, device=device)
    pa.pa_append_decode(pool, q, d["k_new"], d["v_new"], d["bt"], d["sl"], case.scale, out32,
                        partition_blocks=args.partition_blocks, workspace=ws)
    out_fp32 = out32.cpu().numpy()
    code, detail = pa.pa_check(pool)
    assert code == 0, (pa.strerror(code), detail)

    (mean_ms, e2e_ms), total_bytes = reduce_over_ranks([mean_ms, e2e_ms], nbytes["total"], device)
    pool.close()
    return dict(cfg=cfg, case=case, dec_lens=dec_lens, tables=tables, nbytes=nbytes, total_bytes=total_bytes,
                mean_ms=mean_ms,
                p10=float(np.percentile(step_ms, 10)), p90=float(np.percentile(step_ms, 90)),
                median=float(np.median(step_ms)),
                kern_ms=kern_mean, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, wall=wall, clocks=clock_info,
                launches=launches_per_step * K, K=K, l2=flush.l2, out_native=out_native, out_fp32=out_fp32)


def measure_other_configs(args, device):
    """The other workloads, each on its own inputs: the fused step (balanced
    split) and, where the configuration asks for them, fixed partitions
    (long context) and the shared-prefix cascade next to the plain split
    (Llama-2-13B).  Each record keeps the fp32 outputs of one extra call for
    the oracle leg.  K timed steps, L2 flushed before each."""
    import paged_kv_cache_227_gb300 as pa
    peak, _ = measured_peak()
    K, W = max(args.steps, 20), max(args.warmup, 3)
    flush = Flush(device)
    res, keep = {}, {}
    for key in (1, 2, 4, 5):
        _, cfg, case, tables, slots, dec_lens = build_inputs(key, 0, device)
        d = device_inputs(pa, cfg, case, tables, dec_lens, device)
        nb = step_bytes(cfg, dec_lens, tables)
        rec = {"workload": cfg.name, "bytes_per_step": nb["total"], "tokens_attended": int(np.sum(dec_lens))}
        runs = [("balanced", 0)]
        if key == 5:
            longest = int(-(-int(np.max(dec_lens)) // 16))
            runs += [(f"partitions_{P}", -(-longest // P)) for P in (8, 16, 32)]
        outs = {}
        for name, pb in runs:
            out = torch.empty(d["q"].shape, dtype=cfg.torch_dtype, device=device)
            ws = pa.workspace_for(d["pool"], d["q"], d["bt"], pb)
            step = fused_step_fn(pa, d, case, out, pb, ws)
            step_us, kern_us = time_steps(step, flush, K, W, profile=pa)
            kern = float(np.mean(kern_us))
            r = {"partition_blocks": pb, "us_per_step": round(float(np.mean(step_us)), 2),
                 "us_per_step_median": round(float(np.median(step_us)), 2), "kernel_us": round(kern, 2),
                 "kernel_gbs": round(nb["total"] / (kern * 1e-6) / 1e9, 1),
                 "frac_of_copy_peak": round(nb["total"] / (kern * 1e-6) / 1e9 / peak, 4)}
            if name.startswith("partitions"):
                r["partitions_of_longest_sequence"] = int(name.split("_")[1])
            out32 = torch.empty(d["q"].shape, dtype=torch.float32, device=device)
            pa.pa_append_decode(d["pool"], d["q"], d["k_new"], d["v_new"], d["bt"], d["sl"], case.scale, out32,
                                partition_blocks=pb, workspace=ws)
            outs[name] = out32.cpu().numpy()
            rec[name] = r
        code, detail = pa.pa_check(d["pool"])
        assert code == 0, (pa.strerror(code), detail)
        if key == 4:
            # shared prefix: the cascade against the plain balanced split,
            # decode only (the fused steps above wrote the new tokens), L2
            # flushed before each call
            out = torch.empty(d["q"].shape, dtype=cfg.torch_dtype, device=device)
            gs, mem, pre = pa.cascade_groups(tables, dec_lens, cfg.n_q_heads, cfg.n_kv_heads)
            gs_d, mem_d, pre_d = (torch.from_numpy(x).to(device) for x in (gs, mem, pre))
            ws_c = torch.empty(pa.lib.pa_decode_cascade_workspace_bytes(d["pool"].handle, len(dec_lens), cfg.n_q_heads,
                                                                        tables.shape[1], len(pre)),
                               dtype=torch.uint8, device=device)
            ws_s = pa.workspace_for(d["pool"], d["q"], d["bt"], 0)
            calls = {"cascade": lambda o: pa.pa_decode_cascade(d["pool"], d["q"], d["bt"], d["sl"], case.scale, o,
                                                               gs_d, mem_d, pre_d, workspace=ws_c),
                     "plain_split": lambda o: pa.pa_decode_split(d["pool"], d["q"], d["bt"], d["sl"], case.scale, o,
                                                                 0, ws_s)}
            dec_bytes = nb["total"] - nb["new_rows"]
            for name, call in calls.items():
                step_us, _ = time_steps(lambda: call(out), flush, K, W)
                t = float(np.mean(step_us))
                rec[name] = {"us_per_call": round(t, 2), "bytes": dec_bytes,
                             "frac_of_copy_peak": round(dec_bytes / (t * 1e-6) / 1e9 / peak, 4),
                             "note": "decode only (the new tokens are already in the pool); "
                                     "bytes count shared blocks once"}
                out32 = torch.empty(d["q"].shape, dtype=torch.float32, device=device)
                call(out32)
                outs[name] = out32.cpu().numpy()
            rec["cascade"]["groups"] = len(pre)
            code, detail = pa.pa_check(d["pool"])
            assert code == 0, (pa.strerror(code), detail)
        keep[key] = (cfg, case, tables, dec_lens, outs)
        res[str(key)] = rec
        d["pool"].close()
        del d
        torch.cuda.empty_cache()
    return res, keep


class OracleSample:
    """The oracle, as it stands, on the first n (sequence, kv head) groups of
    the step's workload (each group = its G query heads over the sequence's
    appended cache).  Algorithmic bytes of a group: L_i * d * 2 (K, V) * 2."""

    def __init__(self, cfg, case, tables, dec_lens, threads):
        import oracle
        self.oracle = oracle

        def bits(t):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)

        self.q = bits(case.q)
        self.kp, self.vp = oracle.cache.append(bits(case.k_pool), bits(case.v_pool), bits(case.k_new),
                                               bits(case.v_new), self._slots(tables, dec_lens))
        self.cfg, self.case, self.tables, self.lens = cfg, case, tables, dec_lens
        self.code = 0 if cfg.dtype == "fp16" else 1
        self.threads = threads
        self.G = cfg.n_q_heads // cfg.n_kv_heads
        self.groups = len(dec_lens) * cfg.n_kv_heads

    @staticmethod
    def _slots(tables, lens):
        pos = lens.astype(np.int64) - 1
        return tables[np.arange(len(lens)), pos // 16].astype(np.int64) * 16 + pos % 16

    def bytes_of(self, n):
        seq = np.arange(n) // self.cfg.n_kv_heads
        return int(np.sum(self.lens[seq])) * self.cfg.d_head * 2 * 2

    def outputs(self, n):
        """The oracle's output rows of the first n groups (fp64)."""
        rows = np.arange(n * self.G, dtype=np.int32)
        return self.oracle.paged_decode(self.q, self.kp, self.vp, self.code, self.tables, self.lens,
                                        self.case.scale, rows=rows, threads=self.threads)

    def run(self, n, reps=1):
        """Time `reps` passes of the oracle over the first n groups."""
        rows = np.arange(n * self.G, dtype=np.int32)
        t0 = time.perf_counter()
        for _ in range(reps):
            self.oracle.paged_decode(self.q, self.kp, self.vp, self.code, self.tables, self.lens, self.case.scale,
                                     rows=rows, threads=self.threads)
        return time.perf_counter() - t0

    def size_for(self, seconds):
        """(groups, passes) that take about `seconds`: a prefix of the
        groups when the whole workload takes longer, else whole-workload
        passes repeated."""
        n1 = min(self.groups, max(1, 4 * self.threads))
        t1 = self.run(n1)
        n = int(n1 * seconds / max(t1, 1e-6))
        if n < self.groups:
            return max(1, n), 1
        t_all = self.run(self.groups)
        return self.groups, max(1, int(round(seconds / max(t_all, 1e-6))))

    def describe(self, n, reps=1):
        toks = self.bytes_of(n) // (self.cfg.d_head * 4)
        passes = f", {reps} passes" if reps > 1 else ""
        return (f"first {n} of {self.groups} (sequence, kv head) groups, {self.G} q heads each, "
                f"{toks} token rows{passes}; fp64 C oracle, {self.threads} OpenMP threads")


def thread_count_diff(a, b, n):
    """Largest |difference| between two oracle samples' outputs on the first
    n groups (0 when the thread count does not change the result)."""
    return float(np.max(np.abs(a.outputs(n) - b.outputs(n))))


ABS_TOL, REL_TOL = 2e-3, 1e-2  # the parity bar on fp32 output (abs, relative to max |ref|)


def parity_record(got32, ref, got_native=None, dtype=None, v_absmax=None):
    """max |err| of the fp32 output against the fp64 oracle and the pass/fail
    of the bar; for a native 16-bit output, how many elements lie more than
    one 16-bit ulp (plus the kernel's own fp32 error floor) from the rounded
    oracle value."""
    got = np.asarray(got32, np.float64).reshape(ref.shape)
    err = np.abs(got - ref)
    bound = min(ABS_TOL, REL_TOL * float(np.abs(ref).max()))
    rec = {"elements": int(ref.size), "max_abs_err": float(err.max()),
           "max_rel_err": float(err.max() / max(float(np.abs(ref).max()), 1e-30)),
           "tol_abs": ABS_TOL, "tol_rel": REL_TOL, "finite": bool(np.isfinite(got).all()),
           "pass": bool(np.isfinite(got).all() and err.max() <= bound)}
    if got_native is not None:
        r16 = torch.from_numpy(ref).to(torch.float32).to(dtype).to(torch.float64).numpy()
        mant = 7 if dtype == torch.bfloat16 else 10
        min_exp = -126 if dtype == torch.bfloat16 else -14
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r16), 2.0 ** min_exp))) - mant)
        floor = 2e-6 + 2.0 ** -18 * float(v_absmax)
        excess = np.abs(np.asarray(got_native, np.float64).reshape(ref.shape) - r16) - (ulp + floor)
        rec["native_16bit"] = {"max_abs_err": float(np.abs(np.asarray(got_native, np.float64).reshape(ref.shape) - ref).max()),
                               "beyond_one_ulp": int((excess > 0).sum())}
    return rec


def oracle_reference(cfg, case, tables, dec_lens, threads, appended=True):
    """The fp64 oracle's output for a whole workload: over the pool after the
    step's cache write (fused step) or over the pool as cached."""
    import oracle

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    kp, vp = bits(case.k_pool), bits(case.v_pool)
    if appended:
        kp, vp = oracle.cache.append(kp, vp, bits(case.k_new), bits(case.v_new), OracleSample._slots(tables, dec_lens))
    return oracle.paged_decode(bits(case.q), kp, vp, 0 if cfg.dtype == "fp16" else 1, tables, dec_lens, case.scale,
                               threads=threads)


def oracle_leg(line, r, other, other_keep, args):
    """Rank 0 at N=1 only: the fp64 oracle, as it stands, on the host's cores -
    the CPU baseline (a bounded sample of the workload, ~10-30 s), and the
    parity of every measured result against the oracle on its whole
    workload."""
    cfg = r["cfg"]
    threads = len(os.sched_getaffinity(0))
    smp = OracleSample(cfg, r["case"], r["tables"], r["dec_lens"], threads)
    n, reps = smp.size_for(args.cpu_seconds)
    dt = smp.run(n, reps)
    line["cpu_baseline"] = {"value": round(smp.bytes_of(n) * reps / dt / 1e9, 4), "unit": "GB/s",
                            "cores": threads, "kind": "oracle",
                            "sample": smp.describe(n, reps) + f", {dt:.1f} s"}
    # the same oracle on one thread, on a sample sized for about 3 s
    one = OracleSample(cfg, r["case"], r["tables"], r["dec_lens"], 1)
    n1, reps1 = one.size_for(3.0)
    dt1 = one.run(n1, reps1)
    line["cpu_baseline"]["one_thread"] = {"value": round(one.bytes_of(n1) * reps1 / dt1 / 1e9, 4),
                                          "sample": one.describe(n1, reps1) + f", {dt1:.1f} s"}
    # the oracle's result does not depend on its thread count
    n_chk = min(n1, 4 * threads)
    line["cpu_baseline"]["threads_max_abs_diff"] = thread_count_diff(smp, one, n_chk)

    v_absmax = max(float(r["case"].v_pool.float().abs().max()), float(r["case"].v_new.float().abs().max()))
    ref = oracle_reference(cfg, r["case"], r["tables"], r["dec_lens"], threads)
    line["parity"] = parity_record(r["out_fp32"], ref, r["out_native"], cfg.torch_dtype, v_absmax)
    line["parity"]["what"] = ("the timed step (same inputs and launch) with fp32 output vs the fp64 oracle on the whole "
                              "workload; native_16bit: the last timed call's own output")
    for key, (kcfg, kcase, ktables, klens, outs) in (other_keep or {}).items():
        ref_app = oracle_reference(kcfg, kcase, ktables, klens, threads, appended=True)
        for name, got in outs.items():  # (every call ran after the fused steps' cache write)
            other[str(key)][name]["parity"] = parity_record(got, ref_app)


def config_dict(cfg, case, dec_lens, tables, partition_blocks, l2_bytes):
    """The workload description both arms print (identical for the same
    workload)."""
    nb = step_bytes(cfg, dec_lens, tables)
    return {
        "workload": cfg.name,
        "batch_per_gpu": len(dec_lens),
        "n_q_heads": cfg.n_q_heads, "n_kv_heads": cfg.n_kv_heads, "d_head": cfg.d_head,
        "block_size": 16,
        "lengths": "lognormal median 600 sigma 0.8 clip [16,8192] + 1 new token"
        if cfg.key == 3 else str(cfg.lengths),
        "tokens_attended": int(np.sum(dec_lens)),
        "pool_blocks": case.num_blocks,
        "step": "pa_append_decode (append, then balanced split-KV decode and LSE merge as dependent launches)",
        "partition_blocks": partition_blocks,
        "l2": f"flushed before every timed step (read of a {2 * l2_bytes >> 20} MiB buffer)",
        "bytes_per_step": nb,
    }


GB300_L2_BYTES = 129 << 20  # L2 of the part, for the reference arm's config when no GPU is visible


def spawn_ranks(args, n):
    """Start n ranks of this program (one process per GPU) when no launcher
    did; each sees RANK/LOCAL_RANK/WORLD_SIZE/MASTER_* like a torchrun rank."""
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    mp.start_processes(_rank_entry, args=(n, port, sys.argv[1:]), nprocs=n, start_method="spawn", join=True)


def _rank_entry(rank, n, port, argv):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(n),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.argv = [sys.argv[0]] + list(argv)
    main()


def main():
    args = parse()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return spawn_ranks(args, args.gpus)
    rank, world, local = dist_env()
    if world != args.gpus:
        print(json.dumps({"error": f"--gpus {args.gpus} but WORLD_SIZE={world}: launch one rank per GPU"}), flush=True)
        sys.exit(2)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if torch.cuda.device_count() <= local:
        raise SystemExit(f"rank {rank}: needs cuda:{local}, only {torch.cuda.device_count()} GPU(s) visible")
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    if args.row != "decode":
        if rank == 0:
            print(json.dumps(ROWS[args.row](args)), flush=True)
        return
    r = run_ours(args, rank, world, local)
    cfg, nb = r["cfg"], r["nbytes"]
    peak, peak_kind = measured_peak()
    value = r["total_bytes"] / (r["mean_ms"] * 1e-3) / 1e9
    achieved = nb["total"] / (r["kern_ms"] * 1e-3) / 1e9
    traffic = traffic_record(args.workload)
    config = config_dict(cfg, r["case"], r["dec_lens"], r["tables"], args.partition_blocks, r["l2"])
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": r["K"],
        "warmup": args.warmup,
        "ms_per_step": round(r["mean_ms"], 5),
        "us_per_step": round(r["mean_ms"] * 1e3, 2),
        "us_per_step_p10_p90": [round(r["p10"] * 1e3, 2), round(r["p90"] * 1e3, 2)],
        "us_per_step_median": round(r["median"] * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if cfg.dtype == "bf16" else "fp16",
        "data": "synthetic (seeded N(0,1) q/k/v, lengths and random block placement; no dataset)",
        "config": config,
        "roofline": {
            "bound": "hbm",
            "kernel": "append_tail_kernel + decode_kernel + merge_kernel (dependent launches), one step",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "kernel_us": round(r["kern_ms"] * 1e3, 2),
            "traffic": traffic["dram_bytes_per_launch"] if traffic else None,
        },
        "e2e": {
            "value": round(r["total_bytes"] / (r["e2e_ms"] * 1e-3) / 1e9, 1),
            "unit": "GB/s",
            "us_per_step": round(r["e2e_ms"] * 1e3, 2),
            "h2d_bytes_per_step": r["h2d"],
            "d2h_bytes_per_step": r["d2h"],
        },
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if nb["kv_logical"] != nb["kv"]:  # shared blocks: every sequence's own view of its bytes
        line["effective_gbs_logical"] = round(value * (nb["total"] - nb["kv"] + nb["kv_logical"]) / nb["total"], 1)
    other, other_keep = None, None
    if rank == 0 and world == 1 and not args.no_other_configs:
        other, other_keep = measure_other_configs(args, torch.device("cuda", local))
        line["other_configs"] = other
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        oracle_leg(line, r, other, other_keep, args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_multi_query(args):
    """Several new tokens per sequence (speculative verification shape) on the
    workload's sequences: pa_decode_multi, L2 flushed before each call.
    Algorithmic bytes: each sequence's K/V once, plus q and out."""
    import paged_kv_cache_227_gb300 as pa
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    pa_, cfg, case, tables, slots, dec_lens = build_inputs(args.workload, 0, device)
    T = args.new_tokens
    news = np.minimum(dec_lens, T).astype(np.int32)
    q_start = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    n_q = int(q_start[-1])
    pool = pa.Pool(case.num_blocks, cfg.n_kv_heads, cfg.torch_dtype)
    pool.k.copy_(case.k_pool.to(device))
    pool.v.copy_(case.v_pool.to(device))
    g = torch.Generator().manual_seed(5)
    q = torch.randn(n_q, cfg.n_q_heads, cfg.d_head, generator=g).to(cfg.torch_dtype).to(device)
    out = torch.empty_like(q)
    qs, bt, sl = (torch.from_numpy(x).to(device) for x in (q_start, tables, dec_lens))
    ws = torch.empty(pa.lib.pa_decode_multi_workspace_bytes(pool.handle, n_q, len(dec_lens), cfg.n_q_heads,
                                                             tables.shape[1]),
                     dtype=torch.uint8, device=device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush_buf = torch.ones(2 * l2 // 4, dtype=torch.float32, device=device)
    sink = torch.zeros(1, device=device)
    K = max(1, min(args.steps, 2000))
    for _ in range(max(args.warmup, 3)):
        sink.add_(flush_buf.sum())
        pa.pa_decode_multi(pool, q, qs, bt, sl, case.scale, out, workspace=ws)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for k in range(K):
        sink.add_(flush_buf.sum())
        ev[k][0].record()
        pa.pa_decode_multi(pool, q, qs, bt, sl, case.scale, out, workspace=ws)
        ev[k][1].record()
    torch.cuda.synchronize()
    code, detail = pa.pa_check(pool)
    assert code == 0, (pa.strerror(code), detail)
    ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    kv = int(np.sum(dec_lens)) * cfg.n_kv_heads * cfg.d_head * 2 * 2
    nbytes = kv + 2 * n_q * cfg.n_q_heads * cfg.d_head * 2
    peak, _ = measured_peak()
    return {"row": "multi-query", "metric": "paged attention, several new tokens per sequence: GB/s",
            "value": round(nbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "us_per_call": round(ms * 1e3, 2),
            "frac_of_copy_peak": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4), "steps": K,
            "config": {"workload": cfg.name, "new_tokens_per_sequence": T, "query_rows": n_q,
                       "bytes": nbytes, "l2": "flushed before every call"}}


def run_cascade(args):
    """Shared-prefix decode on the Llama-2-13B MHA workload (8 of 16 sequences
    fork one 2,048-token prefix) against the plain balanced split on the same
    inputs; L2 flushed before each call.  Bytes: unique K/V (the shared prefix
    once) plus q and out, so plain decode is scored on the same numerator."""
    import paged_kv_cache_227_gb300 as pa
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    _, cfg, case, tables, slots, dec_lens = build_inputs(4, 0, device)
    pool = pa.Pool(case.num_blocks, cfg.n_kv_heads, cfg.torch_dtype)
    pool.k.copy_(case.k_pool.to(device))
    pool.v.copy_(case.v_pool.to(device))
    q = case.q.to(device)
    out = torch.empty_like(q)
    bt, sl = torch.from_numpy(tables).to(device), torch.from_numpy(dec_lens).to(device)
    gs, mem, pre = pa.cascade_groups(tables, dec_lens, cfg.n_q_heads, cfg.n_kv_heads)
    gs_d, mem_d, pre_d = (torch.from_numpy(x).to(device) for x in (gs, mem, pre))
    ws_c = torch.empty(pa.lib.pa_decode_cascade_workspace_bytes(pool.handle, len(dec_lens), cfg.n_q_heads,
                                                                tables.shape[1], len(pre)),
                       dtype=torch.uint8, device=device)
    ws_s = pa.workspace_for(pool, q, bt, 0)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush_buf = torch.ones(2 * l2 // 4, dtype=torch.float32, device=device)
    sink = torch.zeros(1, device=device)
    calls = {"cascade": lambda: pa.pa_decode_cascade(pool, q, bt, sl, case.scale, out, gs_d, mem_d, pre_d,
                                                     workspace=ws_c),
             "split": lambda: pa.pa_decode_split(pool, q, bt, sl, case.scale, out, 0, ws_s)}
    K = max(1, min(args.steps, 500))
    res = {}
    for name, fn, flush in [(n, f, True) for n, f in calls.items()] + [("split_l2_warm", calls["split"], False)]:
        for _ in range(max(args.warmup, 3)):
            if flush:
                sink.add_(flush_buf.sum())
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for k in range(K):
            if flush:
                sink.add_(flush_buf.sum())
            ev[k][0].record()
            fn()
            ev[k][1].record()
        torch.cuda.synchronize()
        res[name] = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    code, detail = pa.pa_check(pool)
    assert code == 0, (pa.strerror(code), detail)
    tok_bytes = cfg.n_kv_heads * cfg.d_head * 2 * 2
    unique = (int(np.sum(dec_lens)) - int(pre.astype(np.int64) @ (np.diff(gs) - 1)) * 16) * tok_bytes
    nbytes = unique + 2 * q.numel() * 2
    peak, _ = measured_peak()
    return {"row": "cascade", "metric": "shared-prefix decode: unique bytes / time, GB/s",
            "value": round(nbytes / (res["cascade"] * 1e-3) / 1e9, 1), "unit": "GB/s",
            "us_per_call": round(res["cascade"] * 1e3, 2),
            "frac_of_copy_peak": round(nbytes / (res["cascade"] * 1e-3) / 1e9 / peak, 4),
            "plain_split_us": round(res["split"] * 1e3, 2),
            "plain_split_us_without_flush": round(res["split_l2_warm"] * 1e3, 2), "steps": K,
            "config": {"workload": cfg.name, "groups": len(pre), "shared_prefix_blocks": pre.tolist(),
                       "unique_bytes": nbytes, "logical_kv_bytes": int(np.sum(dec_lens)) * tok_bytes,
                       "l2": "flushed before every call"}}


def run_prefix_cache(args):
    """Host allocator: 2,048-token prompts found whole in the prefix cache
    (128 block hashes each) and token-tracked appends."""
    import paged_kv_cache_227_gb300 as pa
    a = pa.BlockAllocator(4096)
    prompt = (np.arange(2048) * 7919 % 50021).astype(np.int32)
    a.seq_add_cached(0, [])
    for t in prompt:
        a.append_token(0, int(t))
    a.seq_free(0)
    n = 200
    t0 = time.perf_counter()
    for s in range(1, n + 1):
        assert a.seq_add_cached(s, prompt) == 2048
        a.seq_free(s)
    dt_lookup = time.perf_counter() - t0
    a.seq_add_cached(n + 1, [])
    t0 = time.perf_counter()
    for k in range(20000):
        a.append_token(n + 1, k)
    dt_append = time.perf_counter() - t0
    return {"row": "prefix-cache", "metric": "prefix-cache lookups: cached blocks found per second (host)",
            "value": round(n * 128 / dt_lookup, 1), "unit": "blocks/s",
            "appends_per_s": round(20000 / dt_append, 1),
            "config": {"prompt_tokens": 2048, "prompts": n, "note": "through the Python binding (one call per prompt)"}}


def run_utilisation(args):
    """Worst-case contiguous reservation vs paging on the 96-block demo and a
    lognormal request stream (host replay)."""
    from paged_kv_cache_227_gb300 import utilization as u
    res = {}
    t0 = time.perf_counter()
    for pol in ("reserve", "paged"):
        tr, adm = u.run(pol, 96, u.demo_requests(), 700)
        res[f"demo_{pol}"] = {"max_running": max(s.running for s in tr), "utilisation": round(u.utilisation(tr), 4),
                              "admitted_at": adm}
    rng = np.random.default_rng(0)
    n = 60
    arr = np.sort(rng.integers(0, 400, n))
    pr = np.clip(np.round(np.exp(np.log(150) + 0.9 * rng.standard_normal(n))), 1, 2000).astype(int)
    outp = np.clip(np.round(np.exp(np.log(200) + 0.8 * rng.standard_normal(n))), 1, 2000).astype(int)
    reqs = [(int(a_), int(p_), int(o_), 2048) for a_, p_, o_ in zip(arr, pr, outp)]
    for pol in ("reserve", "paged"):
        tr, adm = u.run(pol, 1024, reqs, 1500)
        res[f"lognormal_{pol}"] = {"max_running": max(s.running for s in tr),
                                   "utilisation": round(u.utilisation(tr), 4)}
    dt = time.perf_counter() - t0
    return {"row": "utilisation", "metric": "token slots holding tokens / slots held (paged)",
            "value": res["lognormal_paged"]["utilisation"], "unit": "fraction", "results": res,
            "seconds": round(dt, 3)}


ROWS = {"multi-query": run_multi_query, "cascade": run_cascade, "prefix-cache": run_prefix_cache,
        "utilisation": run_utilisation}


def run_reference(args, rank, world):
    """The fp64 CPU oracle as the reference arm: each step runs it on a bounded
    sample of the workload, sized so that warm-up and timed steps together
    take about two minutes; rank 0 alone runs and prints."""
    if rank != 0:
        return
    from oracle.allocator import ReferenceAllocator
    from workloads import CONFIGS, build_tables, make_case
    cfg = CONFIGS[args.workload]
    case = make_case(cfg)
    tables, slots, cows, dec_lens = build_tables(case, ReferenceAllocator(case.num_blocks, 16, case.free_order))
    threads = len(os.sched_getaffinity(0))
    smp = OracleSample(cfg, case, tables, dec_lens, threads)
    n, reps = smp.size_for(min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        smp.run(n, reps)
    dts = [smp.run(n, reps) for _ in range(args.steps)]
    dt = float(np.mean(dts)) if dts else smp.run(n, reps)
    value = smp.bytes_of(n) * reps / dt / 1e9
    l2 = torch.cuda.get_device_properties(0).L2_cache_size if torch.cuda.is_available() else GB300_L2_BYTES
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded N(0,1) q/k/v, lengths and random block placement; no dataset)",
        "config": config_dict(cfg, case, dec_lens, tables, args.partition_blocks, l2),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": smp.describe(n, reps)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


if __name__ == "__main__":
    main()
