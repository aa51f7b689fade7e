"""ctypes front end of the fp64 paged-decode oracle (``paged_attention.c``).

TEST INFRASTRUCTURE (see the package docstring).

Inputs are numpy arrays of raw 16-bit patterns (``np.uint16``) so that fp16
and bf16 reach the C code bit for bit; the C code decodes them to fp64 from
the IEEE definitions.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attention.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lib = None

FP16, BF16 = 0, 1


def build(force=False):
    """Compile ``paged_attention.c`` into ``_liboracle.so`` with gcc (OpenMP if
    the compiler has it).  Building the checker is not using it."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_paged_decode.restype = ctypes.c_int
        lib.oracle_paged_decode.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_long, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int]
        lib.oracle_fp16_to_double.restype = ctypes.c_double
        lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads():
    """Threads the oracle's OpenMP loop can use on this host."""
    return _load().oracle_max_threads()


def fp16_bits_to_double(bits):
    return _load().oracle_fp16_to_double(int(bits))


def bf16_bits_to_double(bits):
    return _load().oracle_bf16_to_double(int(bits))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def paged_decode(q, k_pool, v_pool, dtype, block_tables, seq_lens, scale, rows=None, threads=1):
    """fp64 paged decode attention.

    q        uint16 [B][Hq][d]         (fp16 or bf16 bit patterns)
    k_pool   uint16 [N][Hkv][bs][d]    v_pool likewise
    dtype    0 = fp16, 1 = bf16
    block_tables int32 [B][max_blocks]; seq_lens int32 [B]
    rows     None -> every (seq, head); else flat indices i*Hq + h
    Returns float64 [B][Hq][d] (rows None) or [len(rows)][d].
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k_pool = np.ascontiguousarray(k_pool, dtype=np.uint16)
    v_pool = np.ascontiguousarray(v_pool, dtype=np.uint16)
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, d = q.shape
    N, Hkv, bs, d2 = k_pool.shape
    assert d2 == d and v_pool.shape == k_pool.shape
    assert tables.ndim == 2 and tables.shape[0] == B and lens.shape == (B,)
    if rows is None:
        out = np.zeros((B, Hq, d), np.float64)
        rows_arr, n_rows = None, 0
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int32)
        n_rows = rows_arr.size
        out = np.zeros((n_rows, d), np.float64)
    st = _load().oracle_paged_decode(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), int(dtype), N, bs, Hkv, d,
        _ptr(tables), tables.shape[1], _ptr(lens), B, Hq, float(scale),
        _ptr(rows_arr), n_rows, _ptr(out), int(threads))
    if st != 0:
        raise ValueError(f"oracle_paged_decode failed with status {st}")
    return out
