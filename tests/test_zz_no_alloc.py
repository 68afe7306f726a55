"""The allocation-free decode entry point (pa_decode_no_alloc).

Some callers cannot allocate device memory where they decode (a plug-in
inside a framework that owns all allocations, a serving loop that must not
allocate once running).  pa_decode_no_alloc serves them from a workspace
built into the library.  These tests call it through the C ABI and check it
against pa_decode with a freshly allocated, NaN-filled workspace -- bit for
bit, since both run the same kernels -- and against the oracle.  The built-in
workspace keeps the previous call's contents, so the calls come in a sequence
meant to expose anything stale being read: two calls in a row on a long-context
batch with many partitions, then a different, smaller batch with fewer
partitions and other lengths, twice, then the first batch again.  A batch too
large for the built-in workspace is refused without any GPU work.
"""
import numpy as np
import pytest
import torch

import _cases as C
import paged_kv_cache_302_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu


PT = 512  # partition length of every call here (explicit: PA_DECODE_PARTITION may change the default)


def _setup(w):
    c = C.build_paged(w, check_pool=False)
    tab, ctx = c.dev_tables()
    max_ctx = int(c.ctx.max())
    assert pa.pa_decode_workspace_bytes(w.N, w.H_q, w.H_kv, w.D, max_ctx, PT) <= pa.PA_STATIC_WORKSPACE_BYTES
    qd = C.to_dev(c.q, w.dtype)
    ws = torch.empty(pa.pa_decode_workspace_bytes(w.N, w.H_q, w.H_kv, w.D, max_ctx, PT), dtype=torch.uint8,
                     device="cuda")
    ws.view(torch.int32).fill_(0x7FC00000)          # NaN in every float slot, an absurd value in every int slot
    ref = torch.full((w.N, w.H_q, w.D), float("nan"), device="cuda")
    pa.pa_decode(ref, qd, c.pool, tab, ctx, max_ctx, partition_tokens=PT, workspace=ws)
    torch.cuda.synchronize()
    C.assert_close(ref.cpu().numpy(), C.oracle_decode(c), f"pa_decode {w.name}")
    return c, tab, ctx, max_ctx, qd, ref


def test_no_alloc_matches_pa_decode_bit_for_bit_across_batches():
    long_w = W.yi34b_long(B=16)                     # 8 x 32K: 64 partitions per row, 15 MB of partials
    small_w = W.llama3_8b(n_seqs=64)                # other lengths, mostly 1-4 partitions
    cases = {"long": _setup(long_w), "small": _setup(small_w)}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for name in ("long", "long", "small", "small", "long"):
        c, tab, ctx, max_ctx, qd, ref = cases[name]
        out = torch.full_like(ref, float("nan"))
        pa.pa_decode_no_alloc(out, qd, c.pool, tab, ctx, max_ctx, partition_tokens=PT, dev_err=err)
        torch.cuda.synchronize()
        assert err.item() == 0, f"{name}: device error flags {err.item()}"
        assert torch.equal(out, ref), f"{name}: pa_decode_no_alloc differs from pa_decode"


def test_no_alloc_refuses_a_batch_larger_than_its_workspace():
    L = pa.load()
    N, H_q, H_kv, D, max_ctx = 4096, 32, 8, 128, 8192
    assert pa.pa_decode_workspace_bytes(N, H_q, H_kv, D, max_ctx, 0) > pa.PA_STATIC_WORKSPACE_BYTES
    launches = pa.launch_count()
    st = L.pa_decode_no_alloc(None, 2, None, None, None, None, N, H_q, H_kv, D, 16, 512, 100, max_ctx, 0.088, 0, 1,
                              None, None, None)
    assert st == pa.PA_ERR_UNSUPPORTED
    assert "built-in workspace" in pa.last_error()
    assert pa.launch_count() == launches
