"""The timeout exit of the kernels, made to happen on purpose.

Every wait inside the decode and prefill kernels is bounded; when one runs out
the kernel sets PA_DEV_ERR_TIMEOUT and returns, after letting the copies and
tensor-core products it has already issued land.  pa_set_wait_limit_ns(1) makes
the waits give up almost at once (no fault, no trap: the kernels simply stop
waiting), so these tests drive every CTA through that exit, several calls in a
row, and then check that the call returned, that the flag is set, and that the
next call with the default limit is bit-identical to a clean call made before.
"""
import numpy as np
import pytest
import torch

import _cases as C
import oracle
import paged_kv_cache_302_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu


class short_waits:
    """Context in which every in-kernel wait of new launches gives up after 1 ns."""

    def __enter__(self):
        pa.pa_set_wait_limit_ns(1)

    def __exit__(self, *exc):
        pa.pa_set_wait_limit_ns(0)


@pytest.mark.parametrize("pt", [0, -1])
def test_decode_timeout_exit_flags_returns_and_leaves_the_gpu_usable(pt):
    w = W.llama3_8b(n_seqs=64)
    c = C.build_paged(w, check_pool=False)
    tab, ctx = c.dev_tables()
    qd = C.to_dev(c.q, w.dtype)
    max_ctx = int(c.ctx.max())
    ws = torch.empty(pa.pa_decode_workspace_bytes(w.N, w.H_q, w.H_kv, w.D, max_ctx, pt), dtype=torch.uint8,
                     device="cuda")
    clean = torch.full((w.N, w.H_q, w.D), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode(clean, qd, c.pool, tab, ctx, max_ctx, partition_tokens=pt, workspace=ws, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    with short_waits():
        for _ in range(3):
            out = torch.zeros_like(clean)
            pa.pa_decode(out, qd, c.pool, tab, ctx, max_ctx, partition_tokens=pt, workspace=ws, dev_err=err)
        torch.cuda.synchronize()                       # the calls returned
    assert err.item() & pa.PA_DEV_ERR_TIMEOUT
    err.zero_()
    again = torch.full_like(clean, float("nan"))
    pa.pa_decode(again, qd, c.pool, tab, ctx, max_ctx, partition_tokens=pt, workspace=ws, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(again, clean), "the call after the timed-out ones differs from the clean call"
    pairs = C.sample_pairs(w, 24)
    ref = C.oracle_decode(c, pairs=pairs)
    got = again.cpu().numpy()
    C.assert_close(got[pairs[:, 0], pairs[:, 1]], ref[pairs[:, 0], pairs[:, 1]], "after the timeout exit")


def test_contiguous_decode_timeout_exit():
    w = W.yi34b_long(n_seqs=2, ctx_len=3000, B=16)
    c = C.build_paged(w, check_pool=False)
    tab, ctx = c.dev_tables()
    qd = C.to_dev(c.q, w.dtype)
    S_max = int(c.ctx.max())
    req = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    kb = torch.empty((2, S_max, w.H_kv, w.D), dtype=torch.bfloat16, device="cuda")
    vb = torch.empty_like(kb)
    t = torch.arange(S_max, device="cuda")
    for s in range(w.N):
        phys = tab[s, t // w.B].long()
        kb[req[s]] = c.pool[phys, t % w.B, 0]
        vb[req[s]] = c.pool[phys, t % w.B, 1]
    clean = torch.empty((w.N, w.H_q, w.D), device="cuda")
    pa.pa_decode_contiguous(clean, qd, kb, vb, req, ctx, S_max)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with short_waits():
        out = torch.zeros_like(clean)
        pa.pa_decode_contiguous(out, qd, kb, vb, req, ctx, S_max, dev_err=err)
        torch.cuda.synchronize()
    assert err.item() & pa.PA_DEV_ERR_TIMEOUT
    err.zero_()
    again = torch.zeros_like(clean)
    pa.pa_decode_contiguous(again, qd, kb, vb, req, ctx, S_max, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0 and torch.equal(again, clean)


@pytest.mark.parametrize("kernel", ["wide", "narrow"])
def test_prefill_timeout_exit_flags_returns_and_leaves_the_gpu_usable(kernel, monkeypatch):
    monkeypatch.setenv("PA_PREFILL_KERNEL", kernel)  # each prefill kernel through its exit path
    w = W.llama3_8b(n_seqs=3, grow=1024)
    w.ctx = np.asarray([1500, 700, 1024], dtype=np.int32)
    c = C.build_paged(w, check_pool=False)
    chunks = [1500, 300, 512]
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(q_start[-1])
    q = W.normal_bits(np.random.default_rng(5), (T, w.H_q, w.D), w.dtype)
    qd, qs = C.to_dev(q, w.dtype), torch.from_numpy(q_start).cuda()
    tab, ctx = c.dev_tables()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    clean = torch.full((T, w.H_q, w.D), float("nan"), device="cuda")
    pa.pa_prefill(clean, qd, c.pool, tab, ctx, qs, max(chunks), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    with short_waits():
        for _ in range(3):
            out = torch.zeros_like(clean)
            pa.pa_prefill(out, qd, c.pool, tab, ctx, qs, max(chunks), dev_err=err)
        torch.cuda.synchronize()
    assert err.item() & pa.PA_DEV_ERR_TIMEOUT
    err.zero_()
    again = torch.full_like(clean, float("nan"))
    pa.pa_prefill(again, qd, c.pool, tab, ctx, qs, max(chunks), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(again, clean), "the prefill after the timed-out ones differs from the clean call"
    rows = np.arange(0, T * w.H_q, 97, dtype=np.int32)
    ref = oracle.paged_prefill(q, c.host_pool, c.tables, c.ctx, q_start, w.dtype, rows=rows, nthreads=0)
    got = again.cpu().numpy().reshape(T * w.H_q, w.D)[rows]
    C.assert_close(got, ref.reshape(T * w.H_q, w.D)[rows], "prefill after the timeout exit")
