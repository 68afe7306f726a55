"""Seeded synthetic workloads for the paged-KV decode path.

This module only draws numbers: sequence lengths, free-list permutations and
N(0,1) query / key / value values rounded to 16-bit floats.  It holds none of
the method's arithmetic (no allocation, no attention) and is the one module both
the CUDA path's tests / benchmark and the oracle side take their inputs from.

Shapes follow the workloads the pages discuss (OPT-13B serving, Llama-3-8B and
Yi-34B long-context serving, parallel sampling with a shared prompt); the pages'
datasets (ShareGPT, Alpaca, arXiv-Summarization) are not available, so the
length mixes below stand in for them.

Recipes (seed = 0x5EED + workload index; numpy PCG64 streams):
  tiny        4 seqs, ctx {7, 5, 16, 33}, 2 q heads / 2 KV heads, D 64, B 4,
              fp16, 64 pool blocks; free order starts 7, 1, 3, 5 so the first
              two sequences get the explainer's worked-example tables, the rest
              is a seeded permutation of the other 60 blocks.
  opt13b      64 seqs, ctx ~ U{128..2048}, 40 / 40 heads, D 128, B 16, fp16.
  llama3_8b   256 seqs, ctx = clamp(round(lognormal(ln 1000, 1.0)), 1, 8192),
              32 / 8 heads, D 128, B 16, bf16.
  cow         32 prompts x 1030 tokens, 8 samples each, each sample adds
              U{1..256} tokens; Llama-3-8B head shapes, bf16, B 16.
  yi34b_long  8 seqs x 32768 tokens, 56 / 8 heads, D 128, bf16, B in {8,16,32},
              512-token partitions; also laid out contiguously per request.
All pools get spare blocks for decode growth; the free list of every workload
except ``tiny`` is a seeded permutation of all blocks.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED_BASE = 0x5EED
F16, BF16 = "f16", "bf16"
NAN_BITS = {F16: 0x7E00, BF16: 0x7FC0}   # quiet NaN patterns used to poison unused slots


def round_bits(x, dtype: str) -> np.ndarray:
    """fp32 values -> 16-bit patterns, round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        u = x.view(np.uint32)
        bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
        return ((u + bias) >> 16).astype(np.uint16)
    raise ValueError(dtype)


def bits_to_float(bits, dtype: str) -> np.ndarray:
    """16-bit patterns -> fp32 (for building torch tensors / displays; exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def normal_bits(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    return round_bits(rng.standard_normal(size=shape, dtype=np.float32), dtype)


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    N: int
    H_q: int
    H_kv: int
    D: int
    B: int
    dtype: str
    ctx: np.ndarray                     # [N] int32 context length including the decode token
    NB: int
    free_order: np.ndarray              # [NB] int32, block ids in hand-out order
    partition_tokens: int = 512
    # parallel-sampling fields (cow workload only)
    prompts: int = 0
    samples: int = 0
    prompt_len: int = 0
    extra: np.ndarray | None = None     # [prompts*samples] tokens each sample adds

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def elem_bytes(self) -> int:
        return 2

    @property
    def max_ctx(self) -> int:
        return int(self.ctx.max())

    def max_blocks_per_seq(self, grow: int = 0) -> int:
        return -(-(self.max_ctx + grow) // self.B)

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one decode step reads (valid tokens only)."""
        return int(self.ctx.astype(np.int64).sum()) * 2 * self.H_kv * self.D * self.elem_bytes

    def rng(self, stream: int) -> np.random.Generator:
        """Independent stream per purpose: 0 lengths/order, 1 K/V, 2 q, 3 new tokens, 4+ extra."""
        return np.random.Generator(np.random.PCG64([self.seed, stream]))


def _spare(ctx, B, N, grow):
    return int(np.sum(-(-ctx // B))) + N * (-(-grow // B) + 1) + 64


def tiny() -> Workload:
    seed = SEED_BASE + 0
    ctx = np.array([7, 5, 16, 33], dtype=np.int32)
    NB = 64
    rng = np.random.Generator(np.random.PCG64([seed, 0]))
    head = [7, 1, 3, 5]
    rest = np.array([b for b in range(NB) if b not in head], dtype=np.int32)
    order = np.concatenate([np.array(head, dtype=np.int32), rng.permutation(rest).astype(np.int32)])
    return Workload("tiny", seed, 4, 2, 2, 64, 4, F16, ctx, NB, order)


def opt13b(n_seqs: int = 64, grow: int = 64) -> Workload:
    seed = SEED_BASE + 1
    rng = np.random.Generator(np.random.PCG64([seed, 0]))
    ctx = rng.integers(128, 2048, size=n_seqs, endpoint=True).astype(np.int32)
    NB = _spare(ctx, 16, n_seqs, grow)
    order = rng.permutation(NB).astype(np.int32)
    return Workload("opt13b", seed, n_seqs, 40, 40, 128, 16, F16, ctx, NB, order)


def llama3_8b(n_seqs: int = 256, grow: int = 64, cap: int = 8192) -> Workload:
    seed = SEED_BASE + 2
    rng = np.random.Generator(np.random.PCG64([seed, 0]))
    ln = rng.lognormal(mean=math.log(1000.0), sigma=1.0, size=n_seqs)
    ctx = np.clip(np.rint(ln), 1, cap).astype(np.int32)
    NB = _spare(ctx, 16, n_seqs, grow)
    order = rng.permutation(NB).astype(np.int32)
    return Workload("llama3_8b", seed, n_seqs, 32, 8, 128, 16, BF16, ctx, NB, order)


def cow(prompts: int = 32, samples: int = 8, prompt_len: int = 1030, max_extra: int = 256, grow: int = 64) -> Workload:
    seed = SEED_BASE + 3
    rng = np.random.Generator(np.random.PCG64([seed, 0]))
    extra = rng.integers(1, max_extra, size=prompts * samples, endpoint=True).astype(np.int32)
    ctx = (prompt_len + extra).astype(np.int32)
    B = 16
    shared = prompts * (-(-prompt_len // B))
    private = int(np.sum(-(-ctx // B))) - prompts * samples * (prompt_len // B)
    NB = shared + private + prompts * samples * (-(-grow // B) + 1) + 64
    order = rng.permutation(NB).astype(np.int32)
    return Workload("cow", seed, prompts * samples, 32, 8, 128, B, BF16, ctx, NB, order, prompts=prompts,
                    samples=samples, prompt_len=prompt_len, extra=extra)


def yi34b_long(n_seqs: int = 8, ctx_len: int = 32768, B: int = 16, grow: int = 64) -> Workload:
    seed = SEED_BASE + 4
    rng = np.random.Generator(np.random.PCG64([seed, 0]))
    ctx = np.full(n_seqs, ctx_len, dtype=np.int32)
    NB = _spare(ctx, B, n_seqs, grow)
    order = rng.permutation(NB).astype(np.int32)
    return Workload(f"yi34b_long_B{B}", seed, n_seqs, 56, 8, 128, B, BF16, ctx, NB, order)


def request_ids(w: Workload, n_max: int | None = None) -> np.ndarray:
    """Seeded request-slot ids for the contiguous layout (a permutation of 0..N-1 inside [0, n_max))."""
    n_max = w.N if n_max is None else n_max
    return w.rng(5).permutation(n_max)[: w.N].astype(np.int32)


def queries(w: Workload) -> np.ndarray:
    """[N, H_q, D] query bits for the decode step."""
    return normal_bits(w.rng(2), (w.N, w.H_q, w.D), w.dtype)


def token_kv(w: Workload, n_tokens: int, stream: int = 1):
    """n_tokens rows of K and V bits, each [n_tokens, H_kv, D]."""
    r = w.rng(stream)
    k = normal_bits(r, (n_tokens, w.H_kv, w.D), w.dtype)
    v = normal_bits(r, (n_tokens, w.H_kv, w.D), w.dtype)
    return k, v


def decode_steps(w: Workload, steps: int):
    """Per decode step: new-token K, V [N, H_kv, D] and queries [N, H_q, D]."""
    r = w.rng(6)
    out = []
    for _ in range(steps):
        k = normal_bits(r, (w.N, w.H_kv, w.D), w.dtype)
        v = normal_bits(r, (w.N, w.H_kv, w.D), w.dtype)
        q = normal_bits(r, (w.N, w.H_q, w.D), w.dtype)
        out.append((q, k, v))
    return out


def by_name(name: str, **kw) -> Workload:
    return {"tiny": tiny, "opt13b": opt13b, "llama3_8b": llama3_8b, "cow": cow, "yi34b_long": yi34b_long}[name](**kw)


def beam_search_ops(seed: int = SEED_BASE + 5, prompt_len: int = 37, beams: int = 4, rounds: int = 6,
                    tokens_per_round=(1, 5)):
    """A seeded beam-search schedule as allocator operations.

    Start: one prompt sequence (id 0) of `prompt_len` tokens, forked into `beams` beams.  Each round every live
    beam appends U{tokens_per_round} tokens; then the lowest-ranked half of the beams (a seeded choice) is freed
    and each survivor is forked once, so beams share ever deeper prefixes.  Returns a list of
    ("add", id) / ("append", id, n) / ("fork", parent, child) / ("free", id) / ("round_end", live_ids)."""
    rng = np.random.Generator(np.random.PCG64([seed, 0]))
    ops = [("add", 0), ("append", 0, prompt_len)]
    live, nxt = [0], 1
    for j in range(1, beams):
        ops.append(("fork", 0, nxt))
        live.append(nxt)
        nxt += 1
    for _ in range(rounds):
        for b in live:
            ops.append(("append", b, int(rng.integers(tokens_per_round[0], tokens_per_round[1], endpoint=True))))
        keep = sorted(rng.choice(live, size=max(1, len(live) // 2), replace=False).tolist())
        for b in live:
            if b not in keep:
                ops.append(("free", b))
        live = list(keep)
        for b in keep:
            if len(live) < beams:
                ops.append(("fork", b, nxt))
                live.append(nxt)
                nxt += 1
        ops.append(("round_end", tuple(live)))
    return ops
