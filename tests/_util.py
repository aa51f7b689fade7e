"""Helpers shared by the tests (not by the library or the oracle)."""
import numpy as np
import torch

BS = 16


def bits(t):
    """Raw 16-bit patterns of an fp16/bf16 tensor as np.uint16 (CPU)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def dtype_code(torch_dtype):
    return 0 if torch_dtype == torch.float16 else 1


def pool_from_dense(dense, blocks_per_seq, num_blocks, perm, block_size=BS, fill=0.0):
    """Build a paged pool from per-sequence dense caches without position
    arithmetic: each sequence's [Hkv][L][d] cache is padded to whole blocks,
    cut into block_size-row pieces by numpy reshape, and piece j of sequence i
    is stored at physical block perm[offset_i + j].

    dense: list of float arrays [Hkv][L_i][d].  Returns (pool [N][Hkv][bs][d],
    tables int32 [B][max_blocks] padded with -1)."""
    Hkv, _, d = dense[0].shape
    pool = np.full((num_blocks, Hkv, block_size, d), fill, dtype=np.float64)
    width = max(blocks_per_seq)
    tables = np.full((len(dense), width), -1, dtype=np.int32)
    off = 0
    for i, (x, nb) in enumerate(zip(dense, blocks_per_seq)):
        L = x.shape[1]
        padded = np.full((Hkv, nb * block_size, d), fill, dtype=np.float64)
        padded[:, :L] = x
        pieces = padded.reshape(Hkv, nb, block_size, d).transpose(1, 0, 2, 3)  # [nb][Hkv][bs][d]
        ids = np.asarray(perm[off:off + nb])
        pool[ids] = pieces
        tables[i, :nb] = ids
        off += nb
    return pool, tables


def to_bits(x, torch_dtype):
    """float64 array -> rounded 16-bit tensor and its bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch_dtype)
    return t, bits(t)
