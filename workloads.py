"""Seeded synthetic workloads for paged decode.

This module only draws inputs: sequence lengths, a random physical placement
of blocks, and N(0,1) values for q, the new K/V rows and the pool.  It holds
none of the attention arithmetic and imports neither the CUDA library nor the
oracle, so both can be fed from it.

The pages measure block utilisation on request lengths from two public chat
datasets ("Paged Attention: Managing the KV Cache Like Virtual Memory",
inference-serving tag page); those datasets are not available here, so the
length distributions below (fixed, uniform, lognormal, a shared 2,048-token
prefix) stand in for them.

Seeds: ``torch.Generator().manual_seed(1000 + config)`` for values and the
placement permutation, ``numpy.random.default_rng(1000 + config)`` for
lengths.  Values are drawn in fp32 and rounded to the config's 16-bit type.

Length convention: ``context_lens[i]`` tokens are already cached; a decode
step appends one token per sequence and attends over ``context_lens[i] + 1``.
"""
import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16
HEAD_DIM = 128


@dataclass
class Config:
    key: int
    name: str
    n_q_heads: int
    n_kv_heads: int
    dtype: str                 # "fp16" | "bf16"
    batch: int
    lengths: tuple             # ("fixed", [...]) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi)
    pool_blocks: int = 0       # 0 -> ceil(pool_factor * blocks needed)
    pool_factor: float = 1.25
    shared_prefix: int = 0     # tokens of a common parent prefix
    shared_children: tuple = ()  # sequence indices that fork from the parent
    partition_blocks: tuple = ()  # split-KV partition sizes the config exercises
    d_head: int = HEAD_DIM
    extra: dict = field(default_factory=dict)

    @property
    def group(self):
        return self.n_q_heads // self.n_kv_heads

    @property
    def torch_dtype(self):
        return torch.float16 if self.dtype == "fp16" else torch.bfloat16


CONFIGS = {
    1: Config(1, "tiny-qwen2.5-1.5b-layout-fp16", 12, 2, "fp16", 4,
              ("fixed", [17, 100, 256, 513]), pool_blocks=64),
    2: Config(2, "qwen2.5-1.5b-layout-bf16-b32", 12, 2, "bf16", 32,
              ("uniform", 128, 4096)),
    3: Config(3, "llama3-8b-layout-bf16-b64-lognormal", 32, 8, "bf16", 64,
              ("lognormal", 600.0, 0.8, 16, 8192)),
    4: Config(4, "llama2-13b-layout-mha-fp16-b16-shared-prefix", 40, 40, "fp16", 16,
              ("fixed", [4096] * 16), shared_prefix=2048, shared_children=tuple(range(8))),
    5: Config(5, "llama3-8b-layout-bf16-long-context-split-kv", 32, 8, "bf16", 4,
              ("fixed", [8192, 16384, 24576, 32768]), partition_blocks=(64, 32, 128)),
}


def context_lengths(cfg, seed=None):
    """Cached tokens per sequence before the step (int64 numpy array)."""
    rng = np.random.default_rng(1000 + cfg.key if seed is None else seed)
    kind = cfg.lengths[0]
    if kind == "fixed":
        lens = np.array(cfg.lengths[1], dtype=np.int64)
    elif kind == "uniform":
        _, lo, hi = cfg.lengths
        lens = rng.integers(lo, hi + 1, size=cfg.batch, dtype=np.int64)
    elif kind == "lognormal":
        _, median, sigma, lo, hi = cfg.lengths
        z = rng.standard_normal(cfg.batch)
        lens = np.clip(np.round(np.exp(np.log(median) + sigma * z)), lo, hi).astype(np.int64)
    else:
        raise ValueError(kind)
    assert lens.shape == (cfg.batch,)
    return lens


def blocks_for(tokens):
    """Blocks a sequence of `tokens` tokens occupies (ceil(tokens / 16))."""
    return -(-int(tokens) // BLOCK_SIZE)


def pool_size(cfg, lens):
    if cfg.pool_blocks:
        return cfg.pool_blocks
    need = sum(blocks_for(n + 1) for n in lens)
    if cfg.shared_prefix:
        # children share the parent's prefix blocks; count them once
        shared = cfg.shared_prefix // BLOCK_SIZE
        children = sum(1 for i in cfg.shared_children if i < len(lens))
        need = need - shared * children + shared
    return int(math.ceil(cfg.pool_factor * need))


@dataclass
class Case:
    cfg: Config
    context_lens: np.ndarray   # int64 [B]
    num_blocks: int
    free_order: np.ndarray     # int32 permutation of the pool's blocks
    q: torch.Tensor            # [B][Hq][d]
    k_new: torch.Tensor        # [B][Hkv][d]
    v_new: torch.Tensor
    k_pool: torch.Tensor       # [N][Hkv][16][d]
    v_pool: torch.Tensor
    scale: float


def make_case(cfg_or_key, seed=None, device="cpu", lens=None):
    """Draw every input of one decode step for a config.  Pool contents are
    N(0,1) in every slot (the tables decide which ones are read)."""
    cfg = CONFIGS[cfg_or_key] if isinstance(cfg_or_key, int) else cfg_or_key
    s = 1000 + cfg.key if seed is None else seed
    lens = context_lengths(cfg, s) if lens is None else np.asarray(lens, dtype=np.int64)
    n_blocks = pool_size(cfg, lens)
    gen = torch.Generator().manual_seed(s)
    free_order = torch.randperm(n_blocks, generator=gen).to(torch.int32).numpy()
    B, Hq, Hkv, d = len(lens), cfg.n_q_heads, cfg.n_kv_heads, cfg.d_head

    def randn(*shape):
        return torch.randn(*shape, generator=gen, dtype=torch.float32).to(cfg.torch_dtype).to(device)

    q = randn(B, Hq, d)
    k_new = randn(B, Hkv, d)
    v_new = randn(B, Hkv, d)
    k_pool = randn(n_blocks, Hkv, BLOCK_SIZE, d)
    v_pool = randn(n_blocks, Hkv, BLOCK_SIZE, d)
    return Case(cfg, lens, n_blocks, free_order, q, k_new, v_new, k_pool, v_pool,
                scale=1.0 / math.sqrt(d))


def build_tables(case, allocator):
    """Drive a block allocator through the config's history and return
    (block_tables int32 [B][W] padded with -1, slot_mapping int64 [B] of the
    step's new token, cow list [(src, dst)], decode lengths int32 [B]).

    `allocator` is any object with seq_add / fork / append_slot / table (the
    library's host allocator or the oracle's reference allocator).  Sequence
    ids are 0..B-1; a shared parent, if any, is id B and stays alive so its
    prefix blocks keep a reference."""
    cfg, lens = case.cfg, case.context_lens
    B = len(lens)
    parent = None
    if cfg.shared_prefix:
        parent = B
        allocator.seq_add(parent)
        for _ in range(cfg.shared_prefix):
            allocator.append_slot(parent)
    cows = []
    for i in range(B):
        if parent is not None and i in cfg.shared_children:
            allocator.fork(parent, i)
            n0 = cfg.shared_prefix
        else:
            allocator.seq_add(i)
            n0 = 0
        for _ in range(int(lens[i]) - n0):
            _, cs, cd = allocator.append_slot(i)
            if cs >= 0:
                cows.append((cs, cd))
    slots = np.zeros(B, dtype=np.int64)
    for i in range(B):
        slot, cs, cd = allocator.append_slot(i)
        slots[i] = slot
        if cs >= 0:
            cows.append((cs, cd))
    tables = [allocator.table(i) for i in range(B)]
    width = max(len(t) for t in tables)
    bt = np.full((B, width), -1, dtype=np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = t
    return bt, slots, cows, (lens + 1).astype(np.int32)
