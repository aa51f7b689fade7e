"""Paged KV-cache decode attention for one GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/pa.h``: the functions below
carry the same names as the C entry points and only marshal arguments (torch
tensors -> device pointers, the current torch stream -> cudaStream_t).  Every
step of the computation runs in the library's CUDA kernels; there is no CPU
fallback, and importing fails loudly when the library has not been built.
"""
import ctypes
import os

import torch


_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedattn.so")

PA_FP16, PA_BF16, PA_FP32 = 0, 1, 2
PA_OK = 0
PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_OOM = -1, -2, -3
PA_ERR_CUDA, PA_ERR_DEVICE_CHECK, PA_ERR_TIMEOUT = -4, -5, -6
PA_ERR_SCRATCH_LIMIT = -7
PA_STATIC_SCRATCH_BYTES = 12 << 20
BLOCK_SIZE, HEAD_DIM, MAX_GROUP = 16, 128, 8

_DTYPE_CODE = {torch.float16: PA_FP16, torch.bfloat16: PA_BF16, torch.float32: PA_FP32}
_CODE_DTYPE = {v: k for k, v in _DTYPE_CODE.items()}


class PagedAttentionError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"the CUDA library {LIB_PATH} is not built; run paged_kv_cache_227_gb300.build.build() "
            "(or __graft_entry__.build()) first - there is no fallback")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    sigs = {
        "pa_pool_bytes": (sz, [i32, i32, i32, i32, i32]),
        "pa_pool_create": (i32, [i32, i32, i32, i32, i32, ctypes.POINTER(vp)]),
        "pa_pool_destroy": (i32, [vp]),
        "pa_pool_info": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(sz)]),
        "pa_pool_shape": (i32, [vp] + [ctypes.POINTER(i32)] * 4),
        "pa_cache_append": (i32, [vp, vp, vp, vp, i32, vp]),
        "pa_decode": (i32, [vp, vp, vp, i32, vp, i32, i32, f32, vp, i32, vp]),
        "pa_decode_workspace_bytes": (sz, [vp, i32, i32, i32, i32]),
        "pa_decode_split": (i32, [vp, vp, vp, i32, vp, i32, i32, f32, vp, i32, i32, vp, sz, vp]),
        "pa_append_decode": (i32, [vp, vp, vp, vp, vp, i32, vp, i32, i32, f32, vp, i32, i32, vp, sz, vp]),
        "pa_decode_multi_workspace_bytes": (ctypes.c_size_t, [vp, i32, i32, i32, i32]),
        "pa_decode_multi": (i32, [vp, vp, vp, i32, vp, i32, vp, i32, i32, f32, vp, i32, vp, ctypes.c_size_t, vp]),
        "pa_decode_cascade_workspace_bytes": (ctypes.c_size_t, [vp, i32, i32, i32, i32]),
        "pa_decode_cascade": (i32, [vp, vp, vp, i32, vp, i32, i32, f32, vp, vp, vp, i32, vp, i32, vp,
                                    ctypes.c_size_t, vp]),
        "pa_cascade_groups": (i32, [vp, i32, i32, vp, i32, vp, vp, vp, ctypes.POINTER(i32)]),
        "pa_selftest_wait_timeout": (i32, [vp, ctypes.c_longlong, vp]),
        "pa_decode_split_static": (i32, [vp, vp, vp, i32, vp, i32, i32, f32, vp, i32, i32, vp]),
        "pa_copy_blocks": (i32, [vp, vp, vp, i32, vp]),
        "pa_check": (i32, [vp, vp, ctypes.POINTER(i64)]),
        "pa_profile_start": (i32, [i32]),
        "pa_profile_stop": (i32, [ctypes.POINTER(f32), i32]),
        "pa_strerror": (ctypes.c_char_p, [i32]),
        "pa_alloc_create": (i32, [i32, i32, vp, ctypes.POINTER(vp)]),
        "pa_alloc_destroy": (i32, [vp]),
        "pa_alloc_seq_add": (i32, [vp, i32]),
        "pa_alloc_fork": (i32, [vp, i32, i32]),
        "pa_alloc_append_slot": (i32, [vp, i32, ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_int32)]),
        "pa_alloc_extend": (i32, [vp, i32, i32, vp, ctypes.POINTER(ctypes.c_int32),
                                  ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(i32)]),
        "pa_alloc_seq_free": (i32, [vp, i32]),
        "pa_alloc_table": (i32, [vp, i32, vp, i32, ctypes.POINTER(i32)]),
        "pa_alloc_seq_len": (i32, [vp, i32]),
        "pa_alloc_refcount": (i32, [vp, i32]),
        "pa_alloc_num_free": (i32, [vp]),
        "pa_alloc_seq_add_cached": (i32, [vp, i32, vp, i32, ctypes.POINTER(i32)]),
        "pa_alloc_append_token": (i32, [vp, i32, ctypes.c_int32, ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_int32),
                                        ctypes.POINTER(ctypes.c_int32)]),
        "pa_alloc_block_hash": (i32, [vp, i32, ctypes.POINTER(ctypes.c_uint64)]),
        "pa_alloc_prefix_stats": (i32, [vp, ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i64)]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def strerror(code):
    return lib.pa_strerror(int(code)).decode()


def _check(code, what):
    if code != PA_OK:
        raise PagedAttentionError(code, what)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype=None, device=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be on the GPU")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


class _CudaArray:
    """Exposes a raw device buffer through __cuda_array_interface__ so torch can
    view it without copying."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


class Pool:
    """Owns one pa_pool_t: K and V arrays [num_blocks][n_kv_heads][16][128]."""

    def __init__(self, num_blocks, n_kv_heads, dtype=torch.bfloat16, block_size=BLOCK_SIZE,
                 d_head=HEAD_DIM):
        self._h = ctypes.c_void_p()
        code = lib.pa_pool_create(num_blocks, block_size, n_kv_heads, d_head, _DTYPE_CODE[dtype],
                                  ctypes.byref(self._h))
        _check(code, "pa_pool_create")
        self.num_blocks, self.n_kv_heads, self.dtype = num_blocks, n_kv_heads, dtype
        self.device = torch.device("cuda", torch.cuda.current_device())
        k, v, nbytes = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_size_t()
        _check(lib.pa_pool_info(self._h, ctypes.byref(k), ctypes.byref(v), ctypes.byref(nbytes)), "pa_pool_info")
        self.bytes_per_pool = nbytes.value
        shape = (num_blocks, n_kv_heads, BLOCK_SIZE, HEAD_DIM)
        # views of the library-owned memory (int16 carrier, reinterpreted)
        self.k = torch.as_tensor(_CudaArray(k.value, shape, "<i2"), device=self.device).view(dtype)
        self.v = torch.as_tensor(_CudaArray(v.value, shape, "<i2"), device=self.device).view(dtype)

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            self.k = self.v = None
            lib.pa_pool_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pa_pool_bytes(num_blocks, n_kv_heads, dtype, block_size=BLOCK_SIZE, d_head=HEAD_DIM):
    return lib.pa_pool_bytes(num_blocks, block_size, n_kv_heads, d_head, _DTYPE_CODE[dtype])


def pa_pool_create(num_blocks, block_size, n_kv_heads, d_head, dtype):
    return Pool(num_blocks, n_kv_heads, dtype, block_size, d_head)


def pa_cache_append(pool, k_new, v_new, slot_mapping, stream=None):
    _need(k_new, "k_new", pool.dtype); _need(v_new, "v_new", pool.dtype)
    _need(slot_mapping, "slot_mapping", torch.int64)
    n_tok = slot_mapping.numel()
    if k_new.shape != (n_tok, pool.n_kv_heads, HEAD_DIM) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [n_tok][n_kv_heads][128]")
    _check(lib.pa_cache_append(pool.handle, _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), n_tok,
                               _stream(stream)), "pa_cache_append")


def _decode_args(pool, q, block_tables, seq_lens, out):
    _need(q, "q", pool.dtype); _need(block_tables, "block_tables", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32); _need(out, "out")
    B, Hq, d = q.shape
    if d != HEAD_DIM or block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("shapes: q [B][Hq][128], block_tables [B][W], seq_lens [B]")
    if out.shape != q.shape or out.dtype not in _DTYPE_CODE:
        raise ValueError("out must be [B][Hq][128] of fp16, bf16 or fp32")
    return B, Hq, block_tables.shape[1]


def pa_decode(pool, q, block_tables, seq_lens, scale, out, stream=None):
    B, Hq, W = _decode_args(pool, q, block_tables, seq_lens, out)
    _check(lib.pa_decode(pool.handle, _ptr(q), _ptr(block_tables), W, _ptr(seq_lens), B, Hq,
                         float(scale), _ptr(out), _DTYPE_CODE[out.dtype], _stream(stream)), "pa_decode")


def pa_decode_workspace_bytes(pool, num_seqs, n_q_heads, max_blocks_per_seq, partition_blocks=0):
    return lib.pa_decode_workspace_bytes(pool.handle, num_seqs, n_q_heads, max_blocks_per_seq,
                                         partition_blocks)


def workspace_for(pool, q, block_tables, partition_blocks=0):
    n = pa_decode_workspace_bytes(pool, q.shape[0], q.shape[1], block_tables.shape[1], partition_blocks)
    if n == 0:
        raise PagedAttentionError(PA_ERR_INVALID, "pa_decode_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def pa_decode_split(pool, q, block_tables, seq_lens, scale, out, partition_blocks=0,
                    workspace=None, stream=None):
    B, Hq, W = _decode_args(pool, q, block_tables, seq_lens, out)
    if workspace is None:
        workspace = workspace_for(pool, q, block_tables, partition_blocks)
    _check(lib.pa_decode_split(pool.handle, _ptr(q), _ptr(block_tables), W, _ptr(seq_lens), B, Hq,
                               float(scale), _ptr(out), _DTYPE_CODE[out.dtype], int(partition_blocks),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream)), "pa_decode_split")


def pa_decode_split_static(pool, q, block_tables, seq_lens, scale, out, partition_blocks=0, stream=None):
    """pa_decode_split without a caller workspace: uses the library's static
    device scratch (see include/pa.h); allocates nothing."""
    B, Hq, W = _decode_args(pool, q, block_tables, seq_lens, out)
    _check(lib.pa_decode_split_static(pool.handle, _ptr(q), _ptr(block_tables), W, _ptr(seq_lens), B, Hq,
                                      float(scale), _ptr(out), _DTYPE_CODE[out.dtype], int(partition_blocks),
                                      _stream(stream)), "pa_decode_split_static")


def pa_append_decode(pool, q, k_new, v_new, block_tables, seq_lens, scale, out, partition_blocks=0,
                     workspace=None, stream=None):
    B, Hq, W = _decode_args(pool, q, block_tables, seq_lens, out)
    _need(k_new, "k_new", pool.dtype); _need(v_new, "v_new", pool.dtype)
    if k_new.shape != (B, pool.n_kv_heads, HEAD_DIM) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B][n_kv_heads][128]")
    if workspace is None:
        workspace = workspace_for(pool, q, block_tables, partition_blocks)
    _check(lib.pa_append_decode(pool.handle, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(block_tables), W,
                                _ptr(seq_lens), B, Hq, float(scale), _ptr(out), _DTYPE_CODE[out.dtype],
                                int(partition_blocks), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)),
           "pa_append_decode")


def pa_decode_multi(pool, q, q_start, block_tables, seq_lens, scale, out, workspace=None, stream=None):
    """Several new query tokens per sequence (causal within them); q and out
    are [n_q][Hq][128], q_start int32 [B+1] on the device (see include/pa.h)."""
    _need(q, "q", pool.dtype); _need(q_start, "q_start", torch.int32)
    _need(block_tables, "block_tables", torch.int32); _need(seq_lens, "seq_lens", torch.int32); _need(out, "out")
    n_q, Hq, d = q.shape
    B = seq_lens.shape[0]
    if d != HEAD_DIM or q_start.shape != (B + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("shapes: q [n_q][Hq][128], q_start [B+1], block_tables [B][W], seq_lens [B]")
    if out.shape != q.shape or out.dtype not in _DTYPE_CODE:
        raise ValueError("out must be [n_q][Hq][128] of fp16, bf16 or fp32")
    W = block_tables.shape[1]
    if workspace is None:
        n = lib.pa_decode_multi_workspace_bytes(pool.handle, n_q, B, Hq, W)
        if n == 0:
            raise PagedAttentionError(PA_ERR_INVALID, "pa_decode_multi_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    _check(lib.pa_decode_multi(pool.handle, _ptr(q), _ptr(q_start), n_q, _ptr(block_tables), W, _ptr(seq_lens), B, Hq,
                               float(scale), _ptr(out), _DTYPE_CODE[out.dtype], _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream)), "pa_decode_multi")


def cascade_groups(block_tables, seq_lens, n_q_heads, n_kv_heads):
    """Host: (group_start, members, prefix_blocks) int32 numpy arrays for
    pa_decode_cascade from host tables [B][W] and lengths [B]."""
    import numpy as np
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, W = t.shape
    gs = np.zeros(B + 1, np.int32)
    mem = np.zeros(max(B, 1), np.int32)
    pre = np.zeros(max(B, 1), np.int32)
    ng = ctypes.c_int()
    _check(lib.pa_cascade_groups(t.ctypes.data_as(ctypes.c_void_p), B, W, lens.ctypes.data_as(ctypes.c_void_p),
                                 MAX_GROUP // (n_q_heads // n_kv_heads), gs.ctypes.data_as(ctypes.c_void_p),
                                 mem.ctypes.data_as(ctypes.c_void_p), pre.ctypes.data_as(ctypes.c_void_p),
                                 ctypes.byref(ng)), "pa_cascade_groups")
    n = ng.value
    return gs[:n + 1].copy(), mem[:gs[n]].copy(), pre[:n].copy()


def pa_decode_cascade(pool, q, block_tables, seq_lens, scale, out, group_start, members, prefix_blocks,
                      workspace=None, stream=None):
    """pa_decode with each group's shared prefix read once (include/pa.h);
    the group arrays are int32 device tensors."""
    B, Hq, W = _decode_args(pool, q, block_tables, seq_lens, out)
    for t, n in ((group_start, "group_start"), (members, "members"), (prefix_blocks, "prefix_blocks")):
        _need(t, n, torch.int32)
    ng = prefix_blocks.shape[0]
    if workspace is None:
        n = lib.pa_decode_cascade_workspace_bytes(pool.handle, B, Hq, W, ng)
        if n == 0:
            raise PagedAttentionError(PA_ERR_INVALID, "pa_decode_cascade_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    _check(lib.pa_decode_cascade(pool.handle, _ptr(q), _ptr(block_tables), W, _ptr(seq_lens), B, Hq, float(scale),
                                 _ptr(group_start) if ng else None, _ptr(members) if ng else None,
                                 _ptr(prefix_blocks) if ng else None, ng, _ptr(out), _DTYPE_CODE[out.dtype],
                                 _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "pa_decode_cascade")


def pa_copy_blocks(pool, src, dst, stream=None):
    _need(src, "src", torch.int32); _need(dst, "dst", torch.int32)
    if src.numel() != dst.numel():
        raise ValueError("src and dst must have the same length")
    _check(lib.pa_copy_blocks(pool.handle, _ptr(src), _ptr(dst), src.numel(), _stream(stream)),
           "pa_copy_blocks")


def pa_profile_start(capacity):
    """Time the main decode kernel of the next `capacity` decode calls."""
    _check(lib.pa_profile_start(int(capacity)), "pa_profile_start")


def pa_profile_stop(cap=1 << 20):
    """Milliseconds of each recorded decode kernel (list of floats)."""
    import numpy as np
    buf = np.zeros(max(1, cap), dtype=np.float32)
    n = lib.pa_profile_stop(buf.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), cap)
    if n < 0:
        _check(n, "pa_profile_stop")
    return buf[:min(n, cap)].tolist()


def pa_selftest_wait_timeout(pool, limit_ns, stream=None):
    """Runs the kernels' bounded wait on a barrier nothing arrives at; it gives
    up after limit_ns and records PA_ERR_TIMEOUT (read it with pa_check).
    Returns the launch status."""
    return lib.pa_selftest_wait_timeout(pool.handle, int(limit_ns), _stream(stream))


def pa_check(pool, stream=None):
    """Synchronises the stream and returns (status, detail) of the pool's device
    error word, clearing it."""
    detail = ctypes.c_int64()
    code = lib.pa_check(pool.handle, _stream(stream), ctypes.byref(detail))
    return code, detail.value


class BlockAllocator:
    """The library's host block allocator (pa_alloc_*)."""

    def __init__(self, num_blocks, block_size=BLOCK_SIZE, free_order=None):
        self._h = ctypes.c_void_p()
        arr = None
        if free_order is not None:
            arr = (ctypes.c_int32 * num_blocks)(*[int(b) for b in free_order])
        _check(lib.pa_alloc_create(num_blocks, block_size, arr, ctypes.byref(self._h)), "pa_alloc_create")
        self.num_blocks, self.block_size = num_blocks, block_size

    def __del__(self):
        try:
            if self._h:
                lib.pa_alloc_destroy(self._h)
                self._h = ctypes.c_void_p()
        except Exception:
            pass

    def seq_add(self, seq):
        _check(lib.pa_alloc_seq_add(self._h, seq), "pa_alloc_seq_add")

    def fork(self, parent, child):
        _check(lib.pa_alloc_fork(self._h, parent, child), "pa_alloc_fork")

    def append_slot(self, seq):
        slot, cs, cd = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        code = lib.pa_alloc_append_slot(self._h, seq, ctypes.byref(slot), ctypes.byref(cs), ctypes.byref(cd))
        if code == PA_ERR_OOM:
            raise MemoryError("no free block")
        _check(code, "pa_alloc_append_slot")
        return slot.value, cs.value, cd.value

    def extend(self, seq, n):
        """n appends; returns (slots int64 list, (cow_src, cow_dst))."""
        import numpy as np
        slots = np.zeros(max(n, 1), dtype=np.int64)
        cs, cd, done = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int()
        code = lib.pa_alloc_extend(self._h, seq, n, slots.ctypes.data_as(ctypes.c_void_p), ctypes.byref(cs),
                                   ctypes.byref(cd), ctypes.byref(done))
        if code == PA_ERR_OOM:
            raise MemoryError(f"no free block after {done.value} tokens")
        _check(code, "pa_alloc_extend")
        return slots[:n], (cs.value, cd.value)

    def seq_add_cached(self, seq, tokens):
        """New sequence sharing the cached full blocks of `tokens` (a prompt of
        token ids); returns the number of tokens it now holds."""
        import numpy as np
        arr = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n = ctypes.c_int()
        _check(lib.pa_alloc_seq_add_cached(self._h, seq, arr.ctypes.data_as(ctypes.c_void_p) if arr.size else None,
                                           int(arr.size), ctypes.byref(n)), "pa_alloc_seq_add_cached")
        return n.value

    def append_token(self, seq, token):
        slot, cs, cd = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        code = lib.pa_alloc_append_token(self._h, seq, int(token), ctypes.byref(slot), ctypes.byref(cs),
                                         ctypes.byref(cd))
        if code == PA_ERR_OOM:
            raise MemoryError("no free block")
        _check(code, "pa_alloc_append_token")
        return slot.value, cs.value, cd.value

    def block_hash(self, block):
        h = ctypes.c_uint64()
        r = lib.pa_alloc_block_hash(self._h, block, ctypes.byref(h))
        if r < 0:
            _check(r, "pa_alloc_block_hash")
        return h.value if r == 1 else None

    def prefix_stats(self):
        q, h, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib.pa_alloc_prefix_stats(self._h, ctypes.byref(q), ctypes.byref(h), ctypes.byref(c)),
               "pa_alloc_prefix_stats")
        return q.value, h.value, c.value

    def seq_free(self, seq):
        _check(lib.pa_alloc_seq_free(self._h, seq), "pa_alloc_seq_free")

    def table(self, seq):
        import numpy as np
        n = ctypes.c_int()
        _check(lib.pa_alloc_table(self._h, seq, None, 0, ctypes.byref(n)), "pa_alloc_table")
        out = np.zeros(max(n.value, 1), dtype=np.int32)
        _check(lib.pa_alloc_table(self._h, seq, out.ctypes.data_as(ctypes.c_void_p), n.value, ctypes.byref(n)),
               "pa_alloc_table")
        return out[:n.value].tolist()

    def seq_len(self, seq):
        r = lib.pa_alloc_seq_len(self._h, seq)
        if r < 0:
            _check(r, "pa_alloc_seq_len")
        return r

    def refcount(self, block):
        r = lib.pa_alloc_refcount(self._h, block)
        if r < 0:
            _check(r, "pa_alloc_refcount")
        return r

    def num_free(self):
        return lib.pa_alloc_num_free(self._h)
