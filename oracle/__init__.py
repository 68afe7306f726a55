"""Plain fp64 CPU oracle for the paged-KV decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library never imports, links or executes anything here, and this
package imports nothing from the product package.

Contents
--------
* ``oracle.c`` (built into ``liboracle.so`` with gcc, OpenMP for the timed
  baseline only): 16-bit float decoding, cache write, block copy, the decode
  attention as a plain two-pass fp64 definition (paged and contiguous), the
  explainer's block-streaming pseudocode, split-context partials and their
  merge, and two size formulas.
* ``alloc_model.py``: an independent block-allocator model (free list,
  reference counts, copy-on-write).

Every function cites the page passage it follows; see the docstrings.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
# A prebuilt library to load instead (the mutation tests point this at deliberately broken copies).
_LIB_OVERRIDE = os.environ.get("ORACLE_LIB")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, -O2, OpenMP)."""
    if _LIB_OVERRIDE:
        return _LIB_OVERRIDE
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_half_to_double.restype = dbl
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = dbl
            L.oracle_kv_cache_bytes.argtypes = [dbl] * 5
            L.oracle_kv_cache_bytes.restype = dbl
            L.oracle_tokens_per_page.argtypes = [dbl] * 4
            L.oracle_tokens_per_page.restype = dbl
            L.oracle_reshape_and_cache.argtypes = [P, P, P, P, i32, i32, i32, i32, i32]
            L.oracle_copy_blocks.argtypes = [P, P, i32, i32, i32, i32, i32]
            L.oracle_swap_blocks.argtypes = [P, i32, P, i32, P, i32, ctypes.c_int64]
            L.oracle_paged_decode.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, dbl, i32, P, i32, i32]
            L.oracle_contiguous_decode.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, dbl, i32, P, i32,
                                                   i32]
            L.oracle_paged_prefill.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, dbl, i32, P, i32,
                                               i32]
            L.oracle_paged_decode_online_row.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, dbl, i32]
            L.oracle_paged_partials_row.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, dbl, i32, i32, i32]
            L.oracle_partition_merge.argtypes = [P, P, P, P, P, i32, i32, i32]
            L.oracle_num_threads.argtypes = []
            for name in ("oracle_reshape_and_cache", "oracle_copy_blocks", "oracle_swap_blocks", "oracle_paged_decode",
                         "oracle_contiguous_decode", "oracle_paged_prefill", "oracle_paged_decode_online_row", "oracle_paged_partials_row",
                         "oracle_partition_merge", "oracle_num_threads"):
                getattr(L, name).restype = i32
            del i64
            _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} failed with code {rc}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _dt(dtype) -> int:
    return {"f16": F16, "fp16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16}[dtype] if isinstance(
        dtype, str) else int(dtype)


# --------------------------------------------------------------------------- decoding / sizes

def half_to_double(bits: int) -> float:
    """IEEE binary16 bit pattern -> value (format definition)."""
    return lib().oracle_half_to_double(int(bits) & 0xFFFF)


def bf16_to_double(bits: int) -> float:
    """bfloat16 bit pattern -> value (upper half of a binary32)."""
    return lib().oracle_bf16_to_double(int(bits) & 0xFFFF)


def kv_cache_bytes(tokens, layers, heads, head_dim, elem_bytes=2.0) -> float:
    """PagedAttention explainer, 技術的詳細 / KVキャッシュのメモリ要件: 2 x elem x t x L x H x D_h."""
    return lib().oracle_kv_cache_bytes(tokens, layers, heads, head_dim, elem_bytes)


def tokens_per_page(page_bytes, kv_heads, head_dim, elem_bytes=2.0) -> float:
    """vAttention explainer, 細粒度ページサイズ table: tokens of one layer's K buffer per page."""
    return lib().oracle_tokens_per_page(page_bytes, kv_heads, head_dim, elem_bytes)


# --------------------------------------------------------------------------- cache ops

def reshape_and_cache(k, v, pool, slot_mapping):
    """Write k, v ([T, H_kv, D] uint16 bit patterns) into ``pool`` ([NB, B, 2, H_kv, D], in place)."""
    assert pool.flags.c_contiguous and pool.dtype == np.uint16
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    sm = _c(slot_mapping, np.int64)
    NB, B, two, H_kv, D = pool.shape
    assert two == 2 and k.shape == v.shape and k.shape[1:] == (H_kv, D) and k.shape[0] == sm.shape[0]
    _check(lib().oracle_reshape_and_cache(_ptr(k), _ptr(v), _ptr(pool), _ptr(sm), sm.shape[0], NB, B, H_kv, D),
           "reshape_and_cache")


def copy_blocks(pool, pairs):
    """Copy whole blocks src -> dst for each (src, dst) row of ``pairs`` (in place)."""
    assert pool.flags.c_contiguous and pool.dtype == np.uint16
    pr = _c(pairs, np.int64).reshape(-1, 2)
    NB, B, _, H_kv, D = pool.shape
    _check(lib().oracle_copy_blocks(_ptr(pool), _ptr(pr), pr.shape[0], NB, B, H_kv, D), "copy_blocks")


def swap_blocks(dst_pool, src_pool, pairs):
    """dst_pool[dst] = src_pool[src] for each (src, dst) row of ``pairs`` (in place on dst_pool)."""
    assert dst_pool.flags.c_contiguous and dst_pool.dtype == np.uint16 and src_pool.dtype == np.uint16
    assert dst_pool.shape[1:] == src_pool.shape[1:]
    src_pool = _c(src_pool, np.uint16)
    pr = _c(pairs, np.int64).reshape(-1, 2)
    blk = int(np.prod(dst_pool.shape[1:]))
    _check(lib().oracle_swap_blocks(_ptr(dst_pool), dst_pool.shape[0], _ptr(src_pool), src_pool.shape[0], _ptr(pr),
                                    pr.shape[0], blk), "swap_blocks")


# --------------------------------------------------------------------------- attention

def _pairs(pairs):
    if pairs is None:
        return None, 0
    p = _c(pairs, np.int32).reshape(-1, 2)
    return p, p.shape[0]


def paged_decode(q, pool, tables, ctx, dtype, scale=None, pairs=None, nthreads=1):
    """Two-pass fp64 decode attention through block tables.

    q: [N, H_q, D] uint16 bits; pool: [NB, B, 2, H_kv, D] uint16 bits;
    tables: [N, MB] int32; ctx: [N] int32.  Returns fp64 [N, H_q, D]; when
    ``pairs`` ([n, 2] of (seq, q_head)) is given only those rows are computed
    and the others are NaN.  scale defaults to 1/sqrt(D).
    """
    q = _c(q, np.uint16)
    tables = _c(tables, np.int32)
    ctx = _c(ctx, np.int32)
    N, H_q, D = q.shape
    NB, B, _, H_kv, D2 = pool.shape
    assert D2 == D
    MB = tables.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(float(D))
    out = np.full((N, H_q, D), np.nan, dtype=np.float64)
    pr, npr = _pairs(pairs)
    _check(lib().oracle_paged_decode(_ptr(out), _ptr(q), _ptr(pool), _ptr(tables), _ptr(ctx), N, H_q, H_kv, D, B, MB,
                                     NB, float(scale), _dt(dtype), _ptr(pr) if pr is not None else None, npr,
                                     int(nthreads)), "paged_decode")
    return out


def contiguous_decode(q, kbuf, vbuf, req_ids, ctx, dtype, scale=None, pairs=None, nthreads=1):
    """Two-pass fp64 decode over per-request K/V buffers [N_max, S_max, H_kv, D]."""
    q = _c(q, np.uint16)
    kbuf = _c(kbuf, np.uint16)
    vbuf = _c(vbuf, np.uint16)
    req_ids = _c(req_ids, np.int32)
    ctx = _c(ctx, np.int32)
    N, H_q, D = q.shape
    N_max, S_max, H_kv, D2 = kbuf.shape
    assert D2 == D and vbuf.shape == kbuf.shape
    if scale is None:
        scale = 1.0 / np.sqrt(float(D))
    out = np.full((N, H_q, D), np.nan, dtype=np.float64)
    pr, npr = _pairs(pairs)
    _check(lib().oracle_contiguous_decode(_ptr(out), _ptr(q), _ptr(kbuf), _ptr(vbuf), _ptr(req_ids), _ptr(ctx), N, H_q,
                                          H_kv, D, S_max, N_max, float(scale), _dt(dtype),
                                          _ptr(pr) if pr is not None else None, npr, int(nthreads)),
           "contiguous_decode")
    return out


def paged_prefill(q, pool, tables, ctx, q_start, dtype, scale=None, rows=None, nthreads=1):
    """Causal paged prefill attention, fp64.  q: [T, H_q, D] bits (rows q_start[s]..q_start[s+1]-1 are the
    last tokens of sequence s); returns [T, H_q, D] (only ``rows`` -- flat t*H_q+h indices -- if given)."""
    q = _c(q, np.uint16)
    tables = _c(tables, np.int32)
    ctx = _c(ctx, np.int32)
    q_start = _c(q_start, np.int32)
    T, H_q, D = q.shape
    NB, B, _, H_kv, D2 = pool.shape
    assert D2 == D and q_start.shape[0] == ctx.shape[0] + 1 and q_start[-1] == T
    if scale is None:
        scale = 1.0 / np.sqrt(float(D))
    out = np.full((T, H_q, D), np.nan)
    rr = None if rows is None else _c(rows, np.int32)
    _check(lib().oracle_paged_prefill(_ptr(out), _ptr(q), _ptr(pool), _ptr(tables), _ptr(ctx), _ptr(q_start),
                                      ctx.shape[0], H_q, H_kv, D, B, tables.shape[1], NB, float(scale), _dt(dtype),
                                      _ptr(rr) if rr is not None else None, 0 if rr is None else rr.shape[0],
                                      int(nthreads)), "paged_prefill")
    return out


def paged_decode_online_row(q_row, pool, table_row, ctx, g, dtype, scale=None):
    """The explainer's block-streaming pseudocode for one (sequence, query head)."""
    q_row = _c(q_row, np.uint16)
    table_row = _c(table_row, np.int32)
    NB, B, _, H_kv, D = pool.shape
    if scale is None:
        scale = 1.0 / np.sqrt(float(D))
    out = np.zeros(D, dtype=np.float64)
    _check(lib().oracle_paged_decode_online_row(_ptr(out), _ptr(q_row), _ptr(pool), _ptr(table_row), int(ctx), H_kv, D,
                                                B, NB, int(g), float(scale), _dt(dtype)), "online_row")
    return out


def paged_partials_row(q_row, pool, table_row, ctx, g, dtype, part_tokens, nparts, scale=None):
    """Per-partition (m2, l, acc) of one row; m2 in base-2 units."""
    q_row = _c(q_row, np.uint16)
    table_row = _c(table_row, np.int32)
    NB, B, _, H_kv, D = pool.shape
    if scale is None:
        scale = 1.0 / np.sqrt(float(D))
    m2 = np.zeros(nparts)
    l = np.zeros(nparts)
    acc = np.zeros((nparts, D))
    _check(lib().oracle_paged_partials_row(_ptr(m2), _ptr(l), _ptr(acc), _ptr(q_row), _ptr(pool), _ptr(table_row),
                                           int(ctx), H_kv, D, B, NB, int(g), float(scale), _dt(dtype),
                                           int(part_tokens), int(nparts)), "partials_row")
    return m2, l, acc


def partition_merge(m2, l, acc, nparts):
    """Merge split-context partials: m2, l [R, P]; acc [R, P, D]; nparts [R] -> out [R, D]."""
    m2 = _c(m2, np.float64)
    l = _c(l, np.float64)
    acc = _c(acc, np.float64)
    nparts = _c(nparts, np.int32)
    R, P, D = acc.shape
    out = np.zeros((R, D))
    _check(lib().oracle_partition_merge(_ptr(out), _ptr(m2), _ptr(l), _ptr(acc), _ptr(nparts), R, P, D),
           "partition_merge")
    return out


def num_threads() -> int:
    return lib().oracle_num_threads()
