"""Byte-level models of the cache write and the block copy, and the KV-size
closed form.

TEST INFRASTRUCTURE (see the package docstring).
"""
import numpy as np


def append(k_pool, v_pool, k_new, v_new, slot_mapping, block_size=16):
    """Cache write: token t's K/V rows (all kv heads) go to physical block
    slot // block_size, row slot % block_size; a negative slot is skipped.
    Returns new pool arrays (the inputs are not modified).

    A sequence's cache grows a token at a time into fixed-size blocks
    ("Serving", section 23.4 Paged Attention).
    k_pool/v_pool: any dtype, [N][Hkv][bs][d]; k_new/v_new: [T][Hkv][d]."""
    k_out, v_out = k_pool.copy(), v_pool.copy()
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        block, row = divmod(slot, block_size)
        k_out[block, :, row, :] = k_new[t]
        v_out[block, :, row, :] = v_new[t]
    return k_out, v_out


def copy_blocks(k_pool, v_pool, src, dst):
    """Copy-on-write support: whole block src[j] (all heads, K and V) is
    copied to block dst[j] ("Paged Attention" teaser on the inference-serving
    tag page: sharing with copy-on-write).  Returns new pool arrays."""
    k_out, v_out = k_pool.copy(), v_pool.copy()
    for s, d in zip(np.asarray(src).tolist(), np.asarray(dst).tolist()):
        k_out[d] = k_pool[s]
        v_out[d] = v_pool[s]
    return k_out, v_out


def kv_cache_bytes(n_layers, n_kv_heads, d_head, context_len, batch, n_bytes):
    """KV cache size in bytes, the product of every stored dimension: 2 (keys
    and values) x layers x kv heads x head width x context length x batch x
    bytes per number ("Serving", section 23.1 The Memory Wall)."""
    return 2 * n_layers * n_kv_heads * d_head * context_len * batch * n_bytes


def kv_bytes_per_token(n_layers, n_kv_heads, d_head, n_bytes):
    """Per-token KV size (context length 1, batch 1) of the same product."""
    return kv_cache_bytes(n_layers, n_kv_heads, d_head, 1, 1, n_bytes)
