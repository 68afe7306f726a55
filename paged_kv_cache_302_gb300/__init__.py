"""Paged KV cache decode on one GB300: Python binding of libpa.so (include/pa.h).

The functions below carry the C entry points' names and only marshal
arguments: they read shapes, pointers and the current CUDA stream from torch
tensors and call the library.  Every step of the path runs in the library's
kernels; there is no Python or CPU fallback, and a missing or unloadable
library raises.

Layouts (see include/pa.h): pool [NB, B, 2, H_kv, D]; k, v [T, H_kv, D];
q, out [N, H_q, D]; block_tables [N, MB] int32; ctx_lens [N] int32;
slot_mapping [T] int64; copy pairs [n, 2] int64.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
import threading

import torch

from . import _build

PA_OK, PA_ERR_INVALID, PA_ERR_OOM, PA_ERR_STATE, PA_ERR_CUDA, PA_ERR_UNSUPPORTED = range(6)
PA_F16, PA_BF16, PA_F32 = 0, 1, 2
PA_DEV_ERR_SLOT, PA_DEV_ERR_BLOCK, PA_DEV_ERR_CTX, PA_DEV_ERR_REQ, PA_DEV_ERR_TIMEOUT = 1, 2, 4, 8, 16
_STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID", 2: "PA_ERR_OOM", 3: "PA_ERR_STATE", 4: "PA_ERR_CUDA",
           5: "PA_ERR_UNSUPPORTED"}

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")


class PAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB


def load(build: bool = True) -> ctypes.CDLL:
    """Load libpa.so (compiling it first when it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libpa.so not found at {path}")
            L = ctypes.CDLL(path)
            _declare(L)
            _lib = L
    return _lib


def _declare(L):
    P, i32, i64, sz, f32, u64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float,
                                 ctypes.c_uint64)
    sig = {
        "pa_last_error": ([], ctypes.c_char_p),
        "pa_version": ([], ctypes.c_char_p),
        "pa_launch_count": ([], u64),
        "pa_set_wait_limit_ns": ([u64], None),
        "pa_reshape_and_cache": ([P, P, P, P, i32, i32, i32, i32, i32, i32, P, P], i32),
        "pa_copy_blocks": ([P, P, i32, i32, i32, i32, i32, i32, P, P], i32),
        "pa_decode_workspace_bytes": ([i32, i32, i32, i32, i32, i32], sz),
        "pa_decode": ([P, i32, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32, P, sz, i32, P, P, P],
                      i32),
        "pa_decode_contiguous": ([P, i32, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, f32, i32, P, sz, i32, P, P,
                                  P], i32),
        "pa_partition_reduce": ([P, i32, P, P, P, P, i32, i32, i32, P, P], i32),
        "pa_decode_no_alloc": ([P, i32, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32, i32, P, P, P],
                               i32),
        "pa_alloc_create": ([i32, i32, P, ctypes.POINTER(ctypes.c_void_p)], i32),
        "pa_alloc_destroy": ([P], None),
        "pa_alloc_add_seq": ([P, i32], i32),
        "pa_alloc_append_slots": ([P, i32, i32, P, P, i32, P], i32),
        "pa_alloc_append_batch": ([P, i32, P, P, P, P, i32, P, P, i32, P], i32),
        "pa_update_block_tables": ([P, i32, i32, P, i32, P, P], i32),
        "pa_swap_blocks": ([P, i32, P, i32, P, i32, i32, i32, i32, i32, P, P], i32),
        "pa_write_contiguous": ([P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, P], i32),
        "pa_vkv_create": ([i32, i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_void_p)], i32),
        "pa_vkv_destroy": ([P], None),
        "pa_vkv_info": ([P, P, P, P, P], i32),
        "pa_vkv_alloc_reqid": ([P, P], i32),
        "pa_vkv_step": ([P, P, P, i32], i32),
        "pa_vkv_free_reqid": ([P, i32], i32),
        "pa_vkv_reclaim": ([P], i32),
        "pa_vkv_mapped_pages": ([P, i32, P], i32),
        "pa_prefill": ([P, i32, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32, f32, i32, P, sz, P, P],
                       i32),
        "pa_prefill_workspace_bytes": ([i32, i32, i32, i32, i32], sz),
        "pa_alloc_fork": ([P, i32, i32], i32),
        "pa_alloc_free_seq": ([P, i32], i32),
        "pa_alloc_block_table": ([P, i32, P, i32, P], i32),
        "pa_alloc_block_tables": ([P, i32, P, P, i32, P], i32),
        "pa_alloc_seq_len": ([P, i32, P], i32),
        "pa_alloc_refcount": ([P, i32, P], i32),
        "pa_alloc_num_free": ([P], i32),
        "pa_alloc_free_list": ([P, P, i32, P], i32),
        "pa_alloc_export": ([P, P, sz, ctypes.POINTER(ctypes.c_size_t)], i32),
        "pa_alloc_import": ([P, sz, ctypes.POINTER(ctypes.c_void_p)], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    del i64


def header_functions() -> list[str]:
    """Names of the functions include/pa.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def _check(st: int):
    if st != PA_OK:
        raise PAError(st, load().pa_last_error().decode())


def last_error() -> str:
    return load().pa_last_error().decode()


def version() -> str:
    return load().pa_version().decode()


def launch_count() -> int:
    return int(load().pa_launch_count())


def pa_set_wait_limit_ns(ns: int):
    """Time limit of the in-kernel waits of later launches (0: the built-in 1 s)."""
    load().pa_set_wait_limit_ns(int(ns))


# ----------------------------------------------------------------------------- marshalling helpers

def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float16:
        return PA_F16
    if t == torch.bfloat16:
        return PA_BF16
    if t == torch.float32:
        return PA_F32
    raise PAError(PA_ERR_UNSUPPORTED, f"dtype {t}")


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise PAError(PA_ERR_INVALID, f"{name} must be a tensor")
    if not t.is_cuda:
        raise PAError(PA_ERR_INVALID, f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise PAError(PA_ERR_INVALID, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise PAError(PA_ERR_INVALID, f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _err_ptr(dev_err):
    if dev_err is None:
        return None
    return _dev(dev_err, "dev_err", torch.int32)


def _stream_ptr(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _events_arg(events, stream):
    """Handles of two torch.cuda.Event objects for the library to record.

    torch creates an event's handle lazily and only lets elapsed_time() read
    events it has recorded itself, so both are recorded once here (creating
    them); the library then records them again around the attention kernel,
    which replaces these timestamps."""
    if events is None:
        return None
    s = torch.cuda.current_stream() if stream is None else stream
    for e in events[:2]:
        e.record(s)
    return (ctypes.c_void_p * 2)(events[0].cuda_event, events[1].cuda_event)


# ----------------------------------------------------------------------------- device entry points

def pa_reshape_and_cache(k, v, pool, slot_mapping, dev_err=None, stream=None):
    """Write k, v [T, H_kv, D] into pool [NB, B, 2, H_kv, D] at slot_mapping [T] (int64)."""
    T, H_kv, D = k.shape
    NB, B = pool.shape[0], pool.shape[1]
    if tuple(v.shape) != (T, H_kv, D) or tuple(pool.shape[2:]) != (2, H_kv, D) or k.dtype != pool.dtype:
        raise PAError(PA_ERR_INVALID, "shape/dtype mismatch between k, v and pool")
    if slot_mapping.numel() != T:
        raise PAError(PA_ERR_INVALID, "slot_mapping must have T entries")
    L = load()
    _check(L.pa_reshape_and_cache(_dev(k, "k"), _dev(v, "v", k.dtype), _dev(pool, "pool"),
                                  _dev(slot_mapping, "slot_mapping", torch.int64), T, NB, B, H_kv, D,
                                  _dtype_code(k.dtype), _err_ptr(dev_err), _stream_ptr(stream)))


def pa_copy_blocks(pool, pairs, dev_err=None, stream=None):
    """pool[dst] = pool[src] for each (src, dst) row of pairs [n, 2] (int64, device)."""
    NB, B, _, H_kv, D = pool.shape
    n = pairs.shape[0] if pairs.numel() else 0
    L = load()
    _check(L.pa_copy_blocks(_dev(pool, "pool"), _dev(pairs, "pairs", torch.int64) if n else None, n, NB, B, H_kv, D,
                            _dtype_code(pool.dtype), _err_ptr(dev_err), _stream_ptr(stream)))


def pa_decode_workspace_bytes(N, H_q, H_kv, D, max_ctx, partition_tokens=0) -> int:
    n = load().pa_decode_workspace_bytes(N, H_q, H_kv, D, max_ctx, partition_tokens)
    if n == 0:
        raise PAError(PA_ERR_INVALID, "invalid workspace arguments")
    return int(n)


def _workspace(workspace, nbytes, device):
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise PAError(PA_ERR_INVALID, "workspace too small")
    return workspace


def pa_decode(out, q, pool, block_tables, ctx_lens, max_ctx, scale=None, partition_tokens=0, workspace=None,
              dev_err=None, attend_events=None, stream=None):
    """Paged decode attention: out [N, H_q, D] (fp32 or the KV dtype), on the device or in pinned host memory (the
    kernels then write the rows across the host link: no separate copy of the result)."""
    N, H_q, D = q.shape
    NB, B, _, H_kv, D2 = pool.shape
    MB = block_tables.shape[1]
    if D2 != D or tuple(out.shape) != (N, H_q, D) or q.dtype != pool.dtype:
        raise PAError(PA_ERR_INVALID, "shape/dtype mismatch")
    if tuple(block_tables.shape) != (N, MB) or ctx_lens.numel() != N:
        raise PAError(PA_ERR_INVALID, "block_tables must be [N, MB] and ctx_lens [N]")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    nbytes = pa_decode_workspace_bytes(N, H_q, H_kv, D, int(max_ctx), partition_tokens)
    ws = _workspace(workspace, nbytes, q.device)
    L = load()
    _check(L.pa_decode(_acc(out, "out"), _dtype_code(out.dtype), _dev(q, "q"), _dev(pool, "pool"),
                       _dev(block_tables, "block_tables", torch.int32), _dev(ctx_lens, "ctx_lens", torch.int32), N,
                       H_q, H_kv, D, B, MB, NB, int(max_ctx), scale, int(partition_tokens), _dev(ws, "workspace"),
                       ws.numel() * ws.element_size(), _dtype_code(pool.dtype), _err_ptr(dev_err),
                       _events_arg(attend_events, stream), _stream_ptr(stream)))
    return out


def _acc(t: torch.Tensor, name: str):
    """Pointer of a tensor the GPU can address: a CUDA tensor or a pinned host tensor."""
    if not isinstance(t, torch.Tensor) or not t.is_contiguous():
        raise PAError(PA_ERR_INVALID, f"{name} must be a contiguous tensor")
    if not t.is_cuda and not t.is_pinned():
        raise PAError(PA_ERR_INVALID, f"{name} must be on a CUDA device or in pinned host memory")
    return ctypes.c_void_p(t.data_ptr())


def pa_swap_blocks(dst_pool, src_pool, pairs, dev_err=None, stream=None):
    """dst_pool[dst] = src_pool[src] for (src, dst) rows of pairs [n, 2] int64; pools [NB, B, 2, H_kv, D] on the
    device or in pinned host memory (swap out: device -> host, swap in: host -> device)."""
    NBd, B, _, H_kv, D = dst_pool.shape
    NBs = src_pool.shape[0]
    if tuple(src_pool.shape[1:]) != tuple(dst_pool.shape[1:]) or src_pool.dtype != dst_pool.dtype:
        raise PAError(PA_ERR_INVALID, "pools differ in block shape or dtype")
    if pairs.dtype != torch.int64:
        raise PAError(PA_ERR_INVALID, "pairs must be int64")
    n = pairs.shape[0] if pairs.numel() else 0
    L = load()
    _check(L.pa_swap_blocks(_acc(dst_pool, "dst_pool"), NBd, _acc(src_pool, "src_pool"), NBs,
                            _acc(pairs, "pairs") if n else None, n, B, H_kv, D, _dtype_code(dst_pool.dtype),
                            _err_ptr(dev_err), _stream_ptr(stream)))


def pa_update_block_tables(tables, updates, dev_err=None, stream=None):
    """Apply (row, logical block, physical block) updates [n, 3] (int32, device) to tables [N, MB]."""
    N, MB = tables.shape
    n = updates.shape[0] if updates.numel() else 0
    L = load()
    _check(L.pa_update_block_tables(_dev(tables, "tables", torch.int32), N, MB,
                                    _dev(updates, "updates", torch.int32) if n else None, n, _err_ptr(dev_err),
                                    _stream_ptr(stream)))


PA_STATIC_WORKSPACE_BYTES = 32 * 1024 * 1024


def pa_decode_no_alloc(out, q, pool, block_tables, ctx_lens, max_ctx, scale=None, partition_tokens=0, dev_err=None,
                       attend_events=None, stream=None):
    """pa_decode with the library's built-in workspace: allocates no device memory.

    For callers that cannot allocate device memory where they decode.  The
    batch's workspace must fit in PA_STATIC_WORKSPACE_BYTES; calls that overlap
    on the GPU share (and race on) the one built-in workspace.  The first call
    on a device should come before any stream capture."""
    N, H_q, D = q.shape
    NB, B, _, H_kv, D2 = pool.shape
    MB = block_tables.shape[1]
    if D2 != D or tuple(out.shape) != (N, H_q, D) or q.dtype != pool.dtype:
        raise PAError(PA_ERR_INVALID, "shape/dtype mismatch")
    if tuple(block_tables.shape) != (N, MB) or ctx_lens.numel() != N:
        raise PAError(PA_ERR_INVALID, "block_tables must be [N, MB] and ctx_lens [N]")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    L = load()
    _check(L.pa_decode_no_alloc(_acc(out, "out"), _dtype_code(out.dtype), _dev(q, "q"), _dev(pool, "pool"),
                                _dev(block_tables, "block_tables", torch.int32),
                                _dev(ctx_lens, "ctx_lens", torch.int32), N, H_q, H_kv, D, B, MB, NB, int(max_ctx),
                                scale, int(partition_tokens), _dtype_code(pool.dtype), _err_ptr(dev_err),
                                _events_arg(attend_events, stream), _stream_ptr(stream)))
    return out


def pa_decode_contiguous(out, q, k_buf, v_buf, req_ids, ctx_lens, max_ctx, scale=None, partition_tokens=0,
                         workspace=None, dev_err=None, attend_events=None, stream=None):
    """Decode attention over per-request K/V buffers [N_max, S_max, H_kv, D]."""
    N, H_q, D = q.shape
    N_max, S_max, H_kv, D2 = k_buf.shape
    if D2 != D or tuple(v_buf.shape) != tuple(k_buf.shape) or tuple(out.shape) != (N, H_q, D):
        raise PAError(PA_ERR_INVALID, "shape mismatch")
    if q.dtype != k_buf.dtype or v_buf.dtype != k_buf.dtype:
        raise PAError(PA_ERR_INVALID, "dtype mismatch")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    nbytes = pa_decode_workspace_bytes(N, H_q, H_kv, D, int(max_ctx), partition_tokens)
    ws = _workspace(workspace, nbytes, q.device)
    L = load()
    _check(L.pa_decode_contiguous(_dev(out, "out"), _dtype_code(out.dtype), _dev(q, "q"), _dev(k_buf, "k_buf"),
                                  _dev(v_buf, "v_buf"), _dev(req_ids, "req_ids", torch.int32),
                                  _dev(ctx_lens, "ctx_lens", torch.int32), N, H_q, H_kv, D, N_max, S_max,
                                  int(max_ctx), scale, int(partition_tokens), _dev(ws, "workspace"),
                                  ws.numel() * ws.element_size(), _dtype_code(k_buf.dtype), _err_ptr(dev_err),
                                  _events_arg(attend_events, stream), _stream_ptr(stream)))
    return out


def pa_prefill_workspace_bytes(N, H_kv, D, B, MB) -> int:
    n = load().pa_prefill_workspace_bytes(N, H_kv, D, B, MB)
    if n == 0:
        raise PAError(PA_ERR_INVALID, "invalid prefill workspace arguments")
    return int(n)


def pa_prefill(out, q, pool, block_tables, ctx_lens, q_start, max_q_len, scale=None, workspace=None,
               stage_v=True, dev_err=None, stream=None):
    """Causal paged prefill: q, out [T, H_q, D]; q_start [N+1] int32 (device); chunks are the sequences' last
    tokens, already written to the pool.  A bf16 cache stages V as fp16 in `workspace` (allocated here when None
    and stage_v is true); stage_v=False passes no workspace (P split into two bf16 parts instead)."""
    T, H_q, D = q.shape
    NB, B, _, H_kv, D2 = pool.shape
    N = ctx_lens.numel()
    MB = block_tables.shape[1]
    if D2 != D or tuple(out.shape) != (T, H_q, D) or q.dtype != pool.dtype or q_start.numel() != N + 1:
        raise PAError(PA_ERR_INVALID, "shape/dtype mismatch")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    ws, ws_bytes = None, 0
    if stage_v and pool.dtype == torch.bfloat16:
        ws = _workspace(workspace, pa_prefill_workspace_bytes(N, H_kv, D, B, MB), q.device)
        ws_bytes = ws.numel() * ws.element_size()
    L = load()
    _check(L.pa_prefill(_dev(out, "out"), _dtype_code(out.dtype), _dev(q, "q"), _dev(pool, "pool"),
                        _dev(block_tables, "block_tables", torch.int32), _dev(ctx_lens, "ctx_lens", torch.int32),
                        _dev(q_start, "q_start", torch.int32), N, T, H_q, H_kv, D, B, MB, NB, int(max_q_len), scale,
                        _dtype_code(pool.dtype), _dev(ws, "workspace") if ws is not None else None, ws_bytes,
                        _err_ptr(dev_err), _stream_ptr(stream)))
    return out


def pa_write_contiguous(k, v, k_ptr, v_ptr, req_ids, positions, N_max, S_max, dev_err=None, stream=None):
    """Write k, v [T, H_kv, D] into contiguous buffers (device pointers or tensors [N_max, S_max, H_kv, D])."""
    T, H_kv, D = k.shape

    def ptr(x):
        return _dev(x, "buffer") if isinstance(x, torch.Tensor) else ctypes.c_void_p(int(x))

    L = load()
    _check(L.pa_write_contiguous(_dev(k, "k"), _dev(v, "v", k.dtype), ptr(k_ptr), ptr(v_ptr),
                                 _dev(req_ids, "req_ids", torch.int32), _dev(positions, "positions", torch.int32), T,
                                 int(N_max), int(S_max), H_kv, D, _dtype_code(k.dtype), _err_ptr(dev_err),
                                 _stream_ptr(stream)))


class VirtualKV:
    """pa_vkv_*: virtually contiguous K/V buffers backed by physical pages on demand."""

    def __init__(self, num_layers, max_batch, max_ctx, H_kv, D, dtype=torch.bfloat16):
        self._L = load()
        self._h = ctypes.c_void_p()
        _check(self._L.pa_vkv_create(num_layers, max_batch, max_ctx, H_kv, D, _dtype_code(dtype),
                                     ctypes.byref(self._h)))
        self.layers, self.max_batch, self.H_kv, self.D, self.dtype = num_layers, max_batch, H_kv, D, dtype
        k = (ctypes.c_void_p * num_layers)()
        v = (ctypes.c_void_p * num_layers)()
        S = ctypes.c_int64()
        page = ctypes.c_int64()
        _check(self._L.pa_vkv_info(self._h, k, v, ctypes.byref(S), ctypes.byref(page)))
        self.k_ptrs = [int(x) for x in k]
        self.v_ptrs = [int(x) for x in v]
        self.S = S.value
        self.page_bytes = page.value

    def alloc_reqid(self) -> int:
        r = ctypes.c_int()
        _check(self._L.pa_vkv_alloc_reqid(self._h, ctypes.byref(r)))
        return r.value

    def step(self, req_ids, ctx_lens):
        import numpy as np
        ids = np.ascontiguousarray(req_ids, dtype=np.int32)
        cx = np.ascontiguousarray(ctx_lens, dtype=np.int32)
        _check(self._L.pa_vkv_step(self._h, _i32p(ids), _i32p(cx), len(ids)))

    def free_reqid(self, r: int):
        _check(self._L.pa_vkv_free_reqid(self._h, int(r)))

    def reclaim(self):
        _check(self._L.pa_vkv_reclaim(self._h))

    def mapped_pages(self, r: int) -> int:
        n = ctypes.c_int()
        _check(self._L.pa_vkv_mapped_pages(self._h, int(r), ctypes.byref(n)))
        return n.value

    def close(self):
        if self._h:
            self._L.pa_vkv_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pa_decode_contiguous_raw(out, q, k_ptr: int, v_ptr: int, req_ids, ctx_lens, N_max, S_max, H_kv, max_ctx,
                             scale=None, partition_tokens=0, workspace=None, dev_err=None, attend_events=None,
                             stream=None):
    """pa_decode_contiguous over raw device buffers [N_max, S_max, H_kv, D] of q's dtype (e.g. VirtualKV's)."""
    N, H_q, D = q.shape
    if tuple(out.shape) != (N, H_q, D):
        raise PAError(PA_ERR_INVALID, "shape mismatch")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    nbytes = pa_decode_workspace_bytes(N, H_q, H_kv, D, int(max_ctx), partition_tokens)
    ws = _workspace(workspace, nbytes, q.device)
    L = load()
    _check(L.pa_decode_contiguous(_dev(out, "out"), _dtype_code(out.dtype), _dev(q, "q"), ctypes.c_void_p(int(k_ptr)),
                                  ctypes.c_void_p(int(v_ptr)), _dev(req_ids, "req_ids", torch.int32),
                                  _dev(ctx_lens, "ctx_lens", torch.int32), N, H_q, H_kv, D, int(N_max), int(S_max),
                                  int(max_ctx), scale, int(partition_tokens), _dev(ws, "workspace"),
                                  ws.numel() * ws.element_size(), _dtype_code(q.dtype), _err_ptr(dev_err),
                                  _events_arg(attend_events, stream), _stream_ptr(stream)))
    return out


def pa_partition_reduce(out, part_m2, part_l, part_acc, nparts, dev_err=None, stream=None):
    """Merge split-context partials: m2, l [R, P]; acc [R, P, D]; nparts [R] -> out [R, D]."""
    R, P, D = part_acc.shape
    if tuple(part_m2.shape) != (R, P) or tuple(part_l.shape) != (R, P) or tuple(out.shape) != (R, D):
        raise PAError(PA_ERR_INVALID, "shape mismatch")
    L = load()
    _check(L.pa_partition_reduce(_dev(out, "out"), _dtype_code(out.dtype), _dev(part_m2, "part_m2", torch.float32),
                                 _dev(part_l, "part_l", torch.float32), _dev(part_acc, "part_acc", torch.float32),
                                 _dev(nparts, "nparts", torch.int32), R, P, D, _err_ptr(dev_err),
                                 _stream_ptr(stream)))
    return out


# ----------------------------------------------------------------------------- host allocator

def _i32p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def pa_alloc_create(num_blocks: int, block_size: int, initial_free_order=None):
    import numpy as np
    L = load()
    h = ctypes.c_void_p()
    order = None
    if initial_free_order is not None:
        order = np.ascontiguousarray(initial_free_order, dtype=np.int32)
        if order.shape != (num_blocks,):
            raise PAError(PA_ERR_INVALID, "initial_free_order must have NB entries")
    _check(L.pa_alloc_create(int(num_blocks), int(block_size), _i32p(order) if order is not None else None,
                             ctypes.byref(h)))
    return h


class BlockAllocator:
    """Owner of one pa_alloc handle; methods are the pa_alloc_* calls."""

    def __init__(self, num_blocks: int, block_size: int, initial_free_order=None):
        self.NB = int(num_blocks)
        self.B = int(block_size)
        self._h = pa_alloc_create(num_blocks, block_size, initial_free_order)
        self._L = load()

    def close(self):
        if self._h:
            self._L.pa_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add_seq(self, seq_id: int):
        _check(self._L.pa_alloc_add_seq(self._h, int(seq_id)))

    def append_slots(self, seq_id: int, n: int):
        import numpy as np
        slots = np.zeros(max(n, 1), dtype=np.int64)
        pairs = np.zeros(2, dtype=np.int64)
        ncow = ctypes.c_int(0)
        _check(self._L.pa_alloc_append_slots(self._h, int(seq_id), int(n), _i32p(slots), _i32p(pairs), 1,
                                             ctypes.byref(ncow)))
        return slots[:n], pairs[: 2 * ncow.value].reshape(-1, 2)

    def append_batch(self, seq_ids, n_tokens, table_updates: bool = False):
        """Append n_tokens[i] tokens to seq_ids[i]; returns (slots, cow_pairs) and, with
        table_updates=True, also the [k, 3] int32 (row, logical block, physical block) updates."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        nt = np.ascontiguousarray(n_tokens, dtype=np.int32)
        total = int(nt.sum())
        slots = np.zeros(max(total, 1), dtype=np.int64)
        pairs = np.zeros(2 * max(len(ids), 1), dtype=np.int64)
        ncow = ctypes.c_int(0)
        # entries set per sequence: at most one block per B tokens plus a partial one and a copy
        cap = int((nt // self.B).sum()) + 2 * len(ids) + 1
        upd = np.empty((cap, 3), dtype=np.int32) if table_updates else None
        nupd = ctypes.c_int(0)
        _check(self._L.pa_alloc_append_batch(self._h, len(ids), _i32p(ids), _i32p(nt), _i32p(slots), _i32p(pairs),
                                             max(len(ids), 1), ctypes.byref(ncow),
                                             _i32p(upd) if upd is not None else None, cap, ctypes.byref(nupd)))
        res = (slots[:total], pairs[: 2 * ncow.value].reshape(-1, 2))
        return res + (upd[: nupd.value],) if table_updates else res

    def fork(self, parent: int, child: int):
        _check(self._L.pa_alloc_fork(self._h, int(parent), int(child)))

    def free_seq(self, seq_id: int):
        _check(self._L.pa_alloc_free_seq(self._h, int(seq_id)))

    def block_table(self, seq_id: int):
        import numpy as np
        n = ctypes.c_int(0)
        self._L.pa_alloc_block_table(self._h, int(seq_id), None, 0, ctypes.byref(n))
        out = np.zeros(max(n.value, 1), dtype=np.int32)
        _check(self._L.pa_alloc_block_table(self._h, int(seq_id), _i32p(out), n.value, ctypes.byref(n)))
        return out[: n.value]

    def block_tables(self, seq_ids, MB: int):
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        out = np.zeros((len(ids), MB), dtype=np.int32)
        ctx = np.zeros(len(ids), dtype=np.int32)
        _check(self._L.pa_alloc_block_tables(self._h, len(ids), _i32p(ids), _i32p(out), int(MB), _i32p(ctx)))
        return out, ctx

    def seq_len(self, seq_id: int) -> int:
        v = ctypes.c_int64(0)
        _check(self._L.pa_alloc_seq_len(self._h, int(seq_id), ctypes.byref(v)))
        return v.value

    def refcount(self, block: int) -> int:
        v = ctypes.c_int(0)
        _check(self._L.pa_alloc_refcount(self._h, int(block), ctypes.byref(v)))
        return v.value

    def num_free(self) -> int:
        return int(self._L.pa_alloc_num_free(self._h))

    def free_list(self):
        import numpy as np
        n = self.num_free()
        out = np.zeros(max(n, 1), dtype=np.int32)
        got = ctypes.c_int(0)
        _check(self._L.pa_alloc_free_list(self._h, _i32p(out), n, ctypes.byref(got)))
        return out[: got.value]

    def export_state(self):
        """The whole allocator state as a flat int64 array (pa_alloc_export)."""
        import numpy as np
        n = ctypes.c_size_t(0)
        _check(self._L.pa_alloc_export(self._h, None, 0, ctypes.byref(n)))
        out = np.zeros(max(n.value, 1), dtype=np.int64)
        _check(self._L.pa_alloc_export(self._h, _i32p(out), n.value, ctypes.byref(n)))
        return out[: n.value]

    @classmethod
    def from_state(cls, state):
        """A new allocator rebuilt from an export_state() array (pa_alloc_import, which checks it)."""
        import numpy as np
        a = np.ascontiguousarray(state, dtype=np.int64)
        L = load()
        h = ctypes.c_void_p()
        _check(L.pa_alloc_import(_i32p(a), a.size, ctypes.byref(h)))
        obj = cls.__new__(cls)
        obj.NB, obj.B, obj._h, obj._L = int(a[1]), int(a[2]), h, L
        return obj


__all__ = [name for name in dir() if name.startswith("pa_")] + ["BlockAllocator", "PAError", "load", "version",
                                                                 "launch_count", "header_functions", "last_error"]
