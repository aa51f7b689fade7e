"""fp64 paged attention for several new query tokens per sequence.

TEST INFRASTRUCTURE (see the package docstring).

The step on either side of decode runs attention for several new tokens of a
sequence at once: a chunk of a prompt written onto its blocks, or the drafted
tokens a target model verifies in one pass ("Serving", sections 23.2 Prefill
and Decode and 23.5 Speculative Decoding; the blocks and tables of section
23.4 Paged Attention).  Each new token sees the cached tokens and the new
tokens before it, itself included (causal within the new tokens).

Definition written out (the plainest reading; the pages give no code):
sequence i holds L_i tokens, of which its last T_i = q_start[i+1] - q_start[i]
are the new ones; query row r = q_start[i] + t (t < T_i) sits at position
p = L_i - T_i + t and, for query head h with kv head g = h // (Hq / Hkv),
    out[r][h] = softmax(scale * K_i[g][0..p] q[r][h]) V_i[g][0..p]
with K_i[g][j] = k_pool[table[i][j // 16]][g][j % 16], in fp64 with the
maximum subtracted.  16-bit inputs are decoded exactly (fp16: IEEE half;
bf16: the upper 16 bits of an IEEE single).
"""
import numpy as np

FP16, BF16 = 0, 1


def decode16(bits, dtype):
    """Exact fp64 values of fp16 (dtype 0) or bf16 (dtype 1) bit patterns."""
    bits = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):  # signalling NaN patterns stay NaN
        if dtype == FP16:
            return bits.view(np.float16).astype(np.float64)
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def paged_multi_query(q, k_pool, v_pool, dtype, block_tables, seq_lens, q_start, scale):
    """q uint16 [n_q][Hq][d]; k_pool, v_pool uint16 [N][Hkv][bs][d];
    block_tables int32 [B][W]; seq_lens int32 [B]; q_start int32 [B+1].
    Returns float64 [n_q][Hq][d]."""
    qf = decode16(q, dtype)
    n_q, Hq, d = qf.shape
    N, Hkv, bs, _ = k_pool.shape
    G = Hq // Hkv
    out = np.zeros((n_q, Hq, d))
    for i in range(len(seq_lens)):
        L, r0, r1 = int(seq_lens[i]), int(q_start[i]), int(q_start[i + 1])
        T = r1 - r0
        if T == 0:
            continue
        assert 0 < T <= L, "the new tokens are part of the sequence"
        pos = np.arange(L)
        blocks = np.asarray(block_tables[i])[pos // bs]
        K = decode16(k_pool[blocks, :, pos % bs, :], dtype)   # [L][Hkv][d]
        V = decode16(v_pool[blocks, :, pos % bs, :], dtype)
        Kh = np.repeat(K, G, axis=1).transpose(1, 0, 2)       # [Hq][L][d]
        Vh = np.repeat(V, G, axis=1).transpose(1, 0, 2)
        Q = qf[r0:r1].transpose(1, 0, 2)                      # [Hq][T][d]
        s = scale * (Q @ Kh.transpose(0, 2, 1))                # [Hq][T][L]
        p_t = L - T + np.arange(T)
        s = np.where(pos[None, None, :] <= p_t[None, :, None], s, -np.inf)
        s = s - s.max(axis=2, keepdims=True)
        w = np.exp(s)
        o = (w @ Vh) / w.sum(axis=2, keepdims=True)            # [Hq][T][d]
        out[r0:r1] = o.transpose(1, 0, 2)
    return out
