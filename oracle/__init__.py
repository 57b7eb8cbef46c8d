"""Float64 CPU oracle for the paged-KV attention step — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never imports, links or runs anything here, and nothing here
imports the product: the two share no code.  Inputs for both sides come from
the seeded generators in ``paged_kv_attention_05_gb300.workloads``, which hold
no arithmetic of the method.

Contents:
  * ``oracle.c`` / ``liboracle.so`` — cache write and paged causal attention in
    float64, for bf16 caches and for int8 caches with one scale each (ctypes
    wrappers below);
  * ``blocks.py`` — the block/slot arithmetic the pages print;
  * ``brute.py`` — dense causal attention on contiguous K/V, the textbook form
    the paged oracle must reduce to.

Every function here is pinned by ``tests/test_oracle_*.py`` against values the
pages print, closed forms, invariances and independent library routines.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    """Loads (building first if needed) the float64 oracle library.

    ``ORACLE_LIB`` names another build of ``oracle.c`` to load instead; the
    planted-mistake tests use it to run the pins against altered copies."""
    global _lib
    if _lib is None:
        path = os.environ.get("ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        L.oracle_write.restype = i32
        L.oracle_write.argtypes = [vp, i64, vp, i64, vp, vp, i64, i32, i32, i32, vp, i64]
        L.oracle_attention.restype = i32
        L.oracle_attention.argtypes = [vp, i64, i64, i32, vp, vp, i64, i32, i32, i32,
                                       vp, vp, vp, i64, i64, i32, dbl, vp, i64]
        L.oracle_attention_sampled.restype = i32
        L.oracle_attention_sampled.argtypes = [vp, i64, i64, i32, vp, vp, i64, i32, i32, i32,
                                               vp, vp, vp, i64, i64, i32, dbl, vp, vp, i64, vp]
        f32 = ctypes.c_float
        L.oracle_write_int8.restype = i32
        L.oracle_write_int8.argtypes = [vp, i64, vp, i64, vp, vp, i64, i32, i32, i32, vp, i64,
                                        f32, f32]
        L.oracle_attention_int8.restype = i32
        L.oracle_attention_int8.argtypes = [vp, i64, i64, i32, vp, vp, dbl, dbl, i64, i32, i32,
                                            i32, vp, vp, vp, i64, i64, i32, dbl, vp, i64]
        L.oracle_num_threads.restype = i32
        L.oracle_set_num_threads.argtypes = [i32]
        _lib = L
    return _lib


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _rows(a):
    """Row stride (elements) of an array whose per-row block is contiguous;
    rows themselves may be strided, as in a split of a fused qkv tensor."""
    expect = a.itemsize
    for dim in range(a.ndim - 1, 0, -1):
        assert a.strides[dim] == expect, "per-row block must be contiguous"
        expect *= a.shape[dim]
    return a.strides[0] // a.itemsize


def write(k, v, key_cache, value_cache, slot_mapping):
    """Scatters k/v rows (uint16 bf16 bits, [n, hkv, d], rows may be strided)
    into the caches ([num_blocks, bs, hkv, d] uint16, modified in place).
    Returns the error bits."""
    assert k.dtype == np.uint16 and v.dtype == np.uint16
    assert key_cache.dtype == np.uint16 and key_cache.flags.c_contiguous
    assert value_cache.dtype == np.uint16 and value_cache.flags.c_contiguous
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    nb, bs, hkv, d = key_cache.shape
    n = slot_mapping.shape[0]
    assert k.shape[0] >= n and v.shape[0] >= n
    return lib().oracle_write(_ptr(k), _rows(k), _ptr(v), _rows(v),
                              _ptr(key_cache), _ptr(value_cache), nb, bs, hkv, d,
                              _ptr(slot_mapping), n)


def write_int8(k, v, key_cache, value_cache, slot_mapping, k_scale, v_scale):
    """The cache write into int8 caches ([num_blocks, bs, hkv, d] int8,
    modified in place): code = clamp(rne(x / scale), -127, 127) in fp32.
    Returns the error bits."""
    assert k.dtype == np.uint16 and v.dtype == np.uint16
    assert key_cache.dtype == np.int8 and key_cache.flags.c_contiguous
    assert value_cache.dtype == np.int8 and value_cache.flags.c_contiguous
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    nb, bs, hkv, d = key_cache.shape
    n = slot_mapping.shape[0]
    assert k.shape[0] >= n and v.shape[0] >= n
    return lib().oracle_write_int8(_ptr(k), _rows(k), _ptr(v), _rows(v), _ptr(key_cache),
                                   _ptr(value_cache), nb, bs, hkv, d, _ptr(slot_mapping), n,
                                   float(np.float32(k_scale)), float(np.float32(v_scale)))


def _meta(query_start_loc, seq_lens, block_table):
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    if bt.ndim == 1:
        bt = bt.reshape(1, -1)
    return qsl, sl, bt


def attention(q, key_cache, value_cache, query_start_loc, seq_lens, block_table,
              num_reqs, scale, out=None):
    """Paged causal attention in float64.  q: uint16 [T, hq, d]; returns
    (out float64 [T, hq, d], error bits).  Rows of ``out`` that no valid
    request covers keep their previous contents (NaN for a fresh ``out``)."""
    assert q.dtype == np.uint16 and q.ndim == 3
    T, hq, d = q.shape
    nb, bs, hkv, d2 = key_cache.shape
    assert d == d2
    qsl, sl, bt = _meta(query_start_loc, seq_lens, block_table)
    if out is None:
        out = np.full((T, hq, d), np.nan, dtype=np.float64)
    assert out.dtype == np.float64 and out.flags.c_contiguous and out.shape == (T, hq, d)
    err = lib().oracle_attention(_ptr(q), _rows(q), T, hq, _ptr(key_cache),
                                 _ptr(value_cache), nb, bs, hkv, d, _ptr(qsl), _ptr(sl),
                                 _ptr(bt), bt.shape[1], bt.shape[1], int(num_reqs),
                                 float(scale), _ptr(out), hq * d)
    return out, err


def attention_int8(q, key_cache, value_cache, k_scale, v_scale, query_start_loc, seq_lens,
                   block_table, num_reqs, scale, out=None):
    """Paged causal attention in float64 over int8 caches (K = code * k_scale,
    V = code * v_scale); returns (out float64 [T, hq, d], error bits)."""
    assert q.dtype == np.uint16 and q.ndim == 3
    assert key_cache.dtype == np.int8 and value_cache.dtype == np.int8
    T, hq, d = q.shape
    nb, bs, hkv, d2 = key_cache.shape
    assert d == d2
    qsl, sl, bt = _meta(query_start_loc, seq_lens, block_table)
    if out is None:
        out = np.full((T, hq, d), np.nan, dtype=np.float64)
    assert out.dtype == np.float64 and out.flags.c_contiguous and out.shape == (T, hq, d)
    err = lib().oracle_attention_int8(_ptr(q), _rows(q), T, hq, _ptr(key_cache),
                                      _ptr(value_cache), float(np.float32(k_scale)),
                                      float(np.float32(v_scale)), nb, bs, hkv, d, _ptr(qsl),
                                      _ptr(sl), _ptr(bt), bt.shape[1], bt.shape[1],
                                      int(num_reqs), float(scale), _ptr(out), hq * d)
    return out, err


def attention_sampled(q, key_cache, value_cache, query_start_loc, seq_lens, block_table,
                      num_reqs, scale, rows, heads):
    """The same definition at chosen (row, head) pairs; returns
    (float64 [n_samples, d], error bits)."""
    assert q.dtype == np.uint16 and q.ndim == 3
    T, hq, d = q.shape
    nb, bs, hkv, _ = key_cache.shape
    qsl, sl, bt = _meta(query_start_loc, seq_lens, block_table)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    heads = np.ascontiguousarray(heads, dtype=np.int32)
    out = np.empty((rows.shape[0], d), dtype=np.float64)
    err = lib().oracle_attention_sampled(_ptr(q), _rows(q), T, hq, _ptr(key_cache),
                                         _ptr(value_cache), nb, bs, hkv, d, _ptr(qsl),
                                         _ptr(sl), _ptr(bt), bt.shape[1], bt.shape[1],
                                         int(num_reqs), float(scale), _ptr(rows), _ptr(heads),
                                         rows.shape[0], _ptr(out))
    return out, err


ERR_SLOT_RANGE = 1
ERR_QSL = 2
ERR_SEQ_LEN = 4
ERR_BT_WIDTH = 8
ERR_BLOCK_ID = 16
