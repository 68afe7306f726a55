"""GPU tests of the virtually contiguous KV buffers (pa_vkv_*): pages mapped on demand, deferred
reclamation, the contiguous cache write, and decode over the mapped buffers against the paged path
(bit for bit) and the fp64 oracle."""
import numpy as np
import pytest
import torch

import _cases as C
import oracle
import paged_kv_cache_302_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu


def _pages(n_tokens, row_bytes, page):
    cover = -(-n_tokens // 32) * 32
    return -(-cover * row_bytes // page)


def test_vkv_pages_follow_the_context_and_decode_matches_paged():
    w = W.llama3_8b(n_seqs=3, grow=4096)
    w.ctx = np.array([1500, 4097, 33], dtype=np.int32)
    c = C.build_paged(w)
    V = pa.VirtualKV(1, 4, 6000, w.H_kv, w.D)
    row = w.H_kv * w.D * 2
    if V.page_bytes == 2 * 1024 * 1024:
        # the vAttention explainer's table: Llama-3-8B holds 1024 tokens per 2 MB page of one K buffer
        assert V.page_bytes // row == 1024
    assert V.S >= 6000 and (V.S * row) % V.page_bytes == 0
    reqs = [V.alloc_reqid() for _ in range(w.N)]
    assert sorted(reqs) == [0, 1, 2]
    assert all(V.mapped_pages(r) == 0 for r in reqs)
    V.step(reqs, w.ctx)
    for r, n in zip(reqs, w.ctx):
        assert V.mapped_pages(r) == _pages(int(n), row, V.page_bytes)
    # write every sequence's K/V (as held by the paged pool) at its request slot
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for s in range(w.N):
        n = int(w.ctx[s])
        t = np.arange(n)
        phys = c.tables[s, t // w.B]
        k = np.ascontiguousarray(c.host_pool[phys, t % w.B, 0])
        v = np.ascontiguousarray(c.host_pool[phys, t % w.B, 1])
        pa.pa_write_contiguous(C.to_dev(k, w.dtype), C.to_dev(v, w.dtype), V.k_ptrs[0], V.v_ptrs[0],
                               torch.full((n,), reqs[s], dtype=torch.int32, device="cuda"),
                               torch.arange(n, dtype=torch.int32, device="cuda"), V.max_batch, V.S, dev_err=err)
    req_t = torch.tensor(reqs, dtype=torch.int32, device="cuda")
    ctx_t = torch.from_numpy(w.ctx).cuda()
    for pt in (0, -1):
        out = torch.full((w.N, w.H_q, w.D), float("nan"), device="cuda")
        pa.pa_decode_contiguous_raw(out, C.to_dev(c.q, w.dtype), V.k_ptrs[0], V.v_ptrs[0], req_t, ctx_t, V.max_batch,
                                    V.S, w.H_kv, int(w.ctx.max()), partition_tokens=pt, dev_err=err)
        ref = C.gpu_decode(c, partition_tokens=pt)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert torch.equal(out, ref)
    C.assert_close(out.cpu().numpy(), C.oracle_decode(c), "decode over mapped buffers")
    # growth maps only the new pages; a freed slot keeps its pages for its next owner
    grown = w.ctx + np.array([2000, 0, 1], dtype=np.int32)
    V.step(reqs, grown)
    for r, n in zip(reqs, grown):
        assert V.mapped_pages(r) == _pages(int(n), row, V.page_bytes)
    before = V.mapped_pages(reqs[1])
    V.free_reqid(reqs[1])
    assert V.alloc_reqid() == reqs[1] and V.mapped_pages(reqs[1]) == before
    V.free_reqid(reqs[2])
    V.reclaim()
    assert V.mapped_pages(reqs[2]) == 0 and V.mapped_pages(reqs[1]) == before
    with pytest.raises(pa.PAError):
        V.step([reqs[2]], [10])          # not allocated any more
    with pytest.raises(pa.PAError):
        V.step([reqs[0]], [6001])        # beyond max_ctx
    V.close()


def test_vkv_slots_run_out_cleanly():
    V = pa.VirtualKV(2, 2, 100, 8, 128)
    a, b = V.alloc_reqid(), V.alloc_reqid()
    with pytest.raises(pa.PAError) as e:
        V.alloc_reqid()
    assert e.value.status == pa.PA_ERR_OOM
    V.step([a, b], [100, 1])
    assert V.mapped_pages(a) >= 1 and V.mapped_pages(b) >= 1
    V.close()
