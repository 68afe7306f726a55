"""Scenario builders shared by the GPU tests (not collected by pytest).

Each builder runs the product side (C++ allocator, CUDA kernels through the
C ABI) and the oracle side (allocator model, fp64 C oracle) on the same seeded
inputs from ``workloads`` and checks the bit-exact parts on the way.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
import paged_kv_cache_302_gb300 as pa
import workloads as W
from oracle.alloc_model import AllocModel

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}
ATOL = 2e-3      # max |out - oracle| allowed for fp32 outputs
REL_L2 = 1e-3    # ||out - oracle||_2 / ||oracle||_2 allowed


def to_dev(bits: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()
    return t.view(TORCH_DT[dtype])


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def nan16(dtype: str) -> int:
    return int(np.array([W.NAN_BITS[dtype]], dtype=np.uint16).view(np.int16)[0])


@dataclasses.dataclass
class Paged:
    w: W.Workload
    pool: torch.Tensor            # device [NB, B, 2, H_kv, D]
    host_pool: np.ndarray         # oracle side, uint16 bits
    tables: np.ndarray            # [N, MB] from the C++ allocator (== model's)
    ctx: np.ndarray
    q: np.ndarray                 # [N, H_q, D] bits
    alloc: object = None
    model: object = None

    @property
    def MB(self):
        return self.tables.shape[1]

    def dev_tables(self):
        return torch.from_numpy(self.tables).cuda(), torch.from_numpy(self.ctx.astype(np.int32)).cuda()


def _compare_tables(alloc, model, N, MB):
    tables, ctx = alloc.block_tables(list(range(N)), MB)
    ref = np.full((N, MB), -1, dtype=np.int32)
    for s in range(N):
        t = model.block_table(s)
        ref[s, : len(t)] = t
    assert np.array_equal(tables, ref), "allocator tables differ from the model"
    assert [model.seq_len(s) for s in range(N)] == list(ctx)
    return tables, ctx


def build_paged(w: W.Workload, poison: bool = True, check_pool: bool = True) -> Paged:
    """Allocate every sequence's whole context in order, write all K/V through slot_mapping."""
    alloc = pa.BlockAllocator(w.NB, w.B, w.free_order)
    model = AllocModel(w.NB, w.B, w.free_order)
    got, want = [], []
    for s in range(w.N):
        alloc.add_seq(s)
        model.add_seq(s)
        got.append(alloc.append_slots(s, int(w.ctx[s]))[0])
        want.append(np.asarray(model.append_slots(s, int(w.ctx[s]))[0], dtype=np.int64))
    slots, slots_ref = np.concatenate(got), np.concatenate(want)
    assert np.array_equal(slots, slots_ref), "slot mapping differs from the model"
    tables, ctx = _compare_tables(alloc, model, w.N, w.max_blocks_per_seq())
    k, v = W.token_kv(w, slots.size)
    shape = (w.NB, w.B, 2, w.H_kv, w.D)
    pool = torch.empty(shape, dtype=TORCH_DT[w.dtype], device="cuda")
    pool.view(torch.int16).fill_(nan16(w.dtype) if poison else 0)
    pa.pa_reshape_and_cache(to_dev(k, w.dtype), to_dev(v, w.dtype), pool, torch.from_numpy(slots).cuda())
    host = np.full(shape, W.NAN_BITS[w.dtype] if poison else 0, dtype=np.uint16)
    oracle.reshape_and_cache(k, v, host, slots_ref)
    if check_pool:
        torch.cuda.synchronize()
        assert np.array_equal(to_bits(pool), host), "pool after reshape_and_cache differs from the oracle"
    return Paged(w, pool, host, tables, ctx, W.queries(w), alloc, model)


def build_cow(w: W.Workload, poison: bool = True) -> tuple[Paged, int]:
    """Prompts written once, forked to all samples, then every sample appends its own tokens
    (copy-on-write pairs copied on the device before the new tokens are written)."""
    alloc = pa.BlockAllocator(w.NB, w.B, w.free_order)
    model = AllocModel(w.NB, w.B, w.free_order)
    shape = (w.NB, w.B, 2, w.H_kv, w.D)
    pool = torch.empty(shape, dtype=TORCH_DT[w.dtype], device="cuda")
    pool.view(torch.int16).fill_(nan16(w.dtype) if poison else 0)
    host = np.full(shape, W.NAN_BITS[w.dtype] if poison else 0, dtype=np.uint16)
    # prompts
    p_slots = []
    for p in range(w.prompts):
        base = p * w.samples
        alloc.add_seq(base)
        model.add_seq(base)
        a = alloc.append_slots(base, w.prompt_len)[0]
        assert list(a) == model.append_slots(base, w.prompt_len)[0]
        p_slots.append(a)
        for j in range(1, w.samples):
            alloc.fork(base, base + j)
            model.fork(base, base + j)
    p_slots = np.concatenate(p_slots)
    k, v = W.token_kv(w, p_slots.size, stream=1)
    pa.pa_reshape_and_cache(to_dev(k, w.dtype), to_dev(v, w.dtype), pool, torch.from_numpy(p_slots).cuda())
    oracle.reshape_and_cache(k, v, host, p_slots)
    # divergent tokens: one batched append, copy-on-write, then the writes
    seq_ids = list(range(w.N))
    slots, pairs = alloc.append_batch(seq_ids, w.extra)
    ref_slots, ref_pairs = [], []
    for s in seq_ids:
        a, b = model.append_slots(s, int(w.extra[s]))
        ref_slots += a
        ref_pairs += b
    assert list(slots) == ref_slots and [tuple(r) for r in pairs] == ref_pairs
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(pool, torch.from_numpy(np.ascontiguousarray(pairs)).cuda(), dev_err=err)
    oracle.copy_blocks(host, np.asarray(ref_pairs, dtype=np.int64).reshape(-1, 2))
    k2, v2 = W.token_kv(w, slots.size, stream=7)
    pa.pa_reshape_and_cache(to_dev(k2, w.dtype), to_dev(v2, w.dtype), pool, torch.from_numpy(slots).cuda(),
                            dev_err=err)
    oracle.reshape_and_cache(k2, v2, host, np.asarray(ref_slots, dtype=np.int64))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(to_bits(pool), host), "pool after copy-on-write differs from the oracle"
    tables, ctx = _compare_tables(alloc, model, w.N, w.max_blocks_per_seq())
    return Paged(w, pool, host, tables, ctx, W.queries(w), alloc, model), len(ref_pairs)


def gpu_decode(c: Paged, partition_tokens=0, out_dtype=torch.float32, dev_err=None, q=None):
    w = c.w
    qd = to_dev(c.q if q is None else q, w.dtype)
    out = torch.full((w.N, w.H_q, w.D), float("nan"), dtype=out_dtype, device="cuda")
    tab, ctx = c.dev_tables()
    pa.pa_decode(out, qd, c.pool, tab, ctx, int(c.ctx.max()), partition_tokens=partition_tokens, dev_err=dev_err)
    torch.cuda.synchronize()
    return out


def oracle_decode(c: Paged, pairs=None, nthreads=0):
    return oracle.paged_decode(c.q, c.host_pool, c.tables, c.ctx, c.w.dtype, pairs=pairs, nthreads=nthreads)


def sample_pairs(w: W.Workload, n: int, seed: int = 0) -> np.ndarray:
    """(seq, q_head) pairs: the longest and shortest sequences plus a seeded random sample."""
    rng = np.random.default_rng(seed)
    order = np.argsort(w.ctx)
    seqs = list(order[:2]) + list(order[-2:]) + list(rng.integers(0, w.N, size=max(0, n - 4)))
    heads = rng.integers(0, w.H_q, size=len(seqs))
    heads[: min(4, len(heads))] = [0, w.H_q - 1, w.G - 1 if w.G > 1 else 0, w.H_q // 2][: min(4, len(heads))]
    pairs = np.stack([np.asarray(seqs), heads], axis=1).astype(np.int32)
    _, first = np.unique(pairs, axis=0, return_index=True)
    return pairs[np.sort(first)]


def assert_close(got: np.ndarray, want: np.ndarray, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    d = np.abs(got - want)
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    assert d.max() <= ATOL, f"{what}: max |diff| {d.max():.3e} > {ATOL}"
    assert rel <= REL_L2, f"{what}: rel L2 {rel:.3e} > {REL_L2}"
