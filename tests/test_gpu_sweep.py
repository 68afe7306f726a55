"""Seeded sweeps over the shapes the library supports, every output against the oracle.

Each case draws its shape from a seeded generator -- query heads per KV head G in 1..8, head dim 64 or 128,
block size 4..32, fp16 or bf16, a partition length, 1-9 sequences with lengths from 1 to a few thousand --
builds the pool through the C++ allocator and pa_reshape_and_cache (bit-exact against the oracle's cache
write), and compares every output row of the paged decode, of the contiguous decode over the same K/V, and of
the prefill over random chunks (bf16 both with V staged and with the split P; every fourth shape on the
two-tile prefill kernel), element by element.
"""
import numpy as np
import pytest
import torch

import _cases as C
import oracle
import paged_kv_cache_302_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu


def _random_workload(seed: int, prefill: bool = False) -> W.Workload:
    rng = np.random.default_rng(1000 + seed)
    G = int(rng.integers(1, 9))
    H_kv = int(rng.choice([1, 2, 3, 4, 8]))
    D = int(rng.choice([64, 128]))
    B = int(rng.choice([8, 16, 32] if prefill else [4, 8, 16, 32]))
    dtype = str(rng.choice(["f16", "bf16"]))
    N = int(rng.integers(1, 10))
    top = int(rng.choice([40, 300, 3000]))
    ctx = rng.integers(1, top + 1, size=N).astype(np.int32)
    NB = int(np.sum(-(-ctx // B))) + int(rng.integers(1, 40))
    order = rng.permutation(NB).astype(np.int32)
    return W.Workload(f"sweep{seed}", 2000 + seed, N, G * H_kv, H_kv, D, B, dtype, ctx, NB, order)


@pytest.mark.parametrize("seed", range(32))
def test_decode_sweep_paged_and_contiguous_every_output(seed):
    w = _random_workload(seed)
    c = C.build_paged(w)
    ref = C.oracle_decode(c)
    pt = int(np.random.default_rng(seed).choice([0, -1, 32, 64, 160]))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = C.gpu_decode(c, partition_tokens=pt, dev_err=err)
    assert err.item() == 0
    C.assert_close(out.cpu().numpy(), ref, f"{w.name} G={w.G} D={w.D} B={w.B} {w.dtype} pt={pt}")
    # the same K/V in per-request buffers (request ids a seeded permutation, S_max past the longest context)
    S_max = int(c.ctx.max()) + 7
    req = np.random.default_rng(seed + 1).permutation(w.N).astype(np.int32)
    kb = np.zeros((w.N, S_max, w.H_kv, w.D), dtype=np.uint16)
    vb = np.zeros_like(kb)
    for s in range(w.N):
        n = int(c.ctx[s])
        rows = c.host_pool[c.tables[s, : -(-n // w.B)]].reshape(-1, 2, w.H_kv, w.D)[:n]
        kb[req[s], :n] = rows[:, 0]
        vb[req[s], :n] = rows[:, 1]
    out2 = torch.full_like(out, float("nan"))
    tab, ctx = c.dev_tables()
    pa.pa_decode_contiguous(out2, C.to_dev(c.q, w.dtype), C.to_dev(kb, w.dtype), C.to_dev(vb, w.dtype),
                            torch.from_numpy(req).cuda(), ctx, int(c.ctx.max()), partition_tokens=pt, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out2, out), "contiguous and paged decodes differ"
    ref2 = oracle.contiguous_decode(c.q, kb, vb, req, c.ctx, w.dtype, nthreads=0)
    C.assert_close(out2.cpu().numpy(), ref2, f"{w.name} contiguous")


@pytest.mark.parametrize("seed", range(40))
def test_prefill_sweep_every_output(seed, monkeypatch):
    # every fourth shape on the two-tile kernel, the rest on the default (persistent 2-CTA clusters)
    monkeypatch.setenv("PA_PREFILL_KERNEL", "narrow" if seed % 4 == 3 else "wide")
    w = _random_workload(seed, prefill=True)
    c = C.build_paged(w)
    rng = np.random.default_rng(seed + 7)
    chunks = [int(rng.integers(1, int(n) + 1)) for n in c.ctx]
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(q_start[-1])
    q = W.normal_bits(rng, (T, w.H_q, w.D), w.dtype)
    ref = oracle.paged_prefill(q, c.host_pool, c.tables, c.ctx, q_start, w.dtype, nthreads=0)
    tab, ctx = c.dev_tables()
    for stage_v in ((True, False) if w.dtype == "bf16" else (True,)):
        out = torch.full((T, w.H_q, w.D), float("nan"), device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.pa_prefill(out, C.to_dev(q, w.dtype), c.pool, tab, ctx, torch.from_numpy(q_start).cuda(), max(chunks),
                      stage_v=stage_v, dev_err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        C.assert_close(out.cpu().numpy(), ref,
                       f"{w.name} G={w.G} H_kv={w.H_kv} D={w.D} B={w.B} {w.dtype} stage_v={stage_v}")
