"""The allocation-free decode entry point (pa_decode_no_alloc).

Some callers cannot allocate device memory where they decode (a plug-in
inside a framework that owns all allocations, a serving loop that must not
allocate once running).  pa_decode_no_alloc serves them from a workspace
built into the library.  These tests call it through the C ABI and check it
against pa_decode with a caller-allocated workspace, on two calls in a row
(the built-in workspace keeps the previous call's contents), and check that
a batch too large for the built-in workspace is refused without any GPU work.
"""
import numpy as np
import pytest
import torch

import _cases as C
import paged_kv_cache_302_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [lambda: W.llama3_8b(n_seqs=64), lambda: W.yi34b_long(B=16)],
                         ids=["llama3_8b_64seqs", "yi34b_long"])
def test_no_alloc_matches_pa_decode_on_two_calls_in_a_row(make):
    w = make()
    c = C.build_paged(w, check_pool=False)
    tab, ctx = c.dev_tables()
    max_ctx = int(c.ctx.max())
    assert pa.pa_decode_workspace_bytes(w.N, w.H_q, w.H_kv, w.D, max_ctx, 0) <= pa.PA_STATIC_WORKSPACE_BYTES
    qd = C.to_dev(c.q, w.dtype)
    ref = torch.full((w.N, w.H_q, w.D), float("nan"), device="cuda")
    pa.pa_decode(ref, qd, c.pool, tab, ctx, max_ctx)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        pa.pa_decode_no_alloc(out, qd, c.pool, tab, ctx, max_ctx, dev_err=err)
        torch.cuda.synchronize()
        assert err.item() == 0, f"call {call}: device error flags {err.item()}"
        C.assert_close(out.cpu().numpy(), ref.cpu().numpy().astype(np.float64), f"no-alloc call {call}")


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
