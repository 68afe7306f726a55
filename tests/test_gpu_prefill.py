"""GPU parity of the tcgen05 paged prefill against the fp64 oracle (causal, chunked)."""
import numpy as np
import pytest
import torch

import _cases as C
import oracle
import paged_kv_cache_302_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu


def _run(c, chunks, seed=0, out_dtype=torch.float32, rows=None):
    w = c.w
    rng = np.random.default_rng(seed)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(q_start[-1])
    q = W.normal_bits(rng, (T, w.H_q, w.D), w.dtype)
    tab, ctx = c.dev_tables()
    out = torch.full((T, w.H_q, w.D), float("nan"), dtype=out_dtype, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_prefill(out, C.to_dev(q, w.dtype), c.pool, tab, ctx, torch.from_numpy(q_start).cuda(), int(max(chunks)),
                  dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle.paged_prefill(q, c.host_pool, c.tables, c.ctx, q_start, w.dtype, rows=rows, nthreads=0)
    return out, ref, q, q_start


def _with_ctx(w, ctx):
    w.ctx = np.asarray(ctx, dtype=np.int32)
    return w


@pytest.mark.parametrize("chunks_of", ["full", "tail", "mixed"])
def test_prefill_llama_shaped_every_output(chunks_of):
    w = _with_ctx(W.llama3_8b(n_seqs=4), [200, 513, 77, 1000])
    c = C.build_paged(w)
    chunks = {"full": list(w.ctx), "tail": [1, 1, 1, 1], "mixed": [200, 130, 1, 257]}[chunks_of]
    out, ref, _, _ = _run(c, chunks)
    C.assert_close(out.cpu().numpy(), ref, f"prefill {chunks_of}")


@pytest.mark.parametrize("make,ctx,chunks", [
    (lambda: W.opt13b(n_seqs=3), [300, 129, 700], [300, 50, 129]),         # MHA, fp16
    (lambda: W.yi34b_long(n_seqs=2, ctx_len=600, B=8), [600, 331], [600, 200]),   # G = 7, B = 8
    (lambda: W.yi34b_long(n_seqs=2, ctx_len=600, B=32), [600, 331], [333, 331]),  # B = 32
])
def test_prefill_group_sizes_and_block_sizes(make, ctx, chunks):
    c = C.build_paged(_with_ctx(make(), ctx))
    out, ref, _, _ = _run(c, chunks)
    C.assert_close(out.cpu().numpy(), ref, f"prefill {c.w.name}")


def test_prefill_head_dim_64():
    w = W.Workload("d64", 1, 3, 8, 2, 64, 8, "f16", np.array([100, 9, 256], np.int32), 200,
                   np.random.default_rng(3).permutation(200).astype(np.int32))
    c = C.build_paged(w)
    out, ref, _, _ = _run(c, [100, 9, 129])
    C.assert_close(out.cpu().numpy(), ref, "prefill D=64")


def test_prefill_one_token_chunks_match_decode():
    w = W.llama3_8b(n_seqs=16)
    c = C.build_paged(w)
    out, ref, q, _ = _run(c, [1] * w.N)
    dec = C.gpu_decode(c, q=q.reshape(w.N, w.H_q, w.D))
    C.assert_close(out.cpu().numpy(), ref, "one-token prefill")
    C.assert_close(out.cpu().numpy(), dec.cpu().numpy().astype(np.float64), "prefill vs decode")


def test_prefill_large_chunks_sampled_rows():
    w = _with_ctx(W.llama3_8b(n_seqs=6, grow=4096), [4096, 3000, 2048, 4096, 1500, 2600])
    c = C.build_paged(w, check_pool=False)
    chunks = [2048, 3000, 1024, 512, 1500, 1]
    rng = np.random.default_rng(11)
    T = sum(chunks)
    rows = np.unique(np.concatenate([rng.integers(0, T * w.H_q, size=200), [0, T * w.H_q - 1]])).astype(np.int32)
    out, ref, _, _ = _run(c, chunks, rows=rows)
    o = out.cpu().numpy().reshape(-1, w.D)[rows]
    C.assert_close(o, ref.reshape(-1, w.D)[rows], "prefill large")
    assert np.all(np.isfinite(out.cpu().numpy()))


@pytest.mark.parametrize("make,ctx,chunks", [
    (lambda: W.llama3_8b(n_seqs=3), [300, 129, 700], [300, 50, 129]),    # bf16
    (lambda: W.opt13b(n_seqs=2), [200, 513], [200, 77]),                  # fp16
], ids=["bf16", "fp16"])
def test_prefill_low_precision_output_is_the_rounded_fp32_output(make, ctx, chunks):
    """A 16-bit prefill output is the round-to-nearest-even of the fp32 output of the same inputs, bit for bit."""
    c = C.build_paged(_with_ctx(make(), ctx))
    w = c.w
    out32, ref, _, _ = _run(c, chunks)
    odt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    out16, _, _, _ = _run(c, chunks, out_dtype=odt)
    bits = C.to_bits(out16)
    assert np.array_equal(bits, W.round_bits(out32.cpu().numpy(), w.dtype))
    half_ulp = np.abs(W.bits_to_float(bits + 1, w.dtype) - W.bits_to_float(bits, w.dtype)) / 2
    assert np.all(np.abs(W.bits_to_float(bits, w.dtype) - ref) <= C.ATOL + half_ulp)


def test_prefill_device_errors_are_flagged_not_faulted():
    """A block id outside the pool is flagged (its copy reads zeros) and a chunk longer than its context is flagged
    and not computed; the context stays usable and the next call is exact."""
    w = _with_ctx(W.llama3_8b(n_seqs=3), [300, 129, 700])
    c = C.build_paged(w)
    chunks = [300, 50, 129]
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(q_start[-1])
    q = W.normal_bits(np.random.default_rng(0), (T, w.H_q, w.D), w.dtype)
    tab, ctx = c.dev_tables()
    out = torch.zeros((T, w.H_q, w.D), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_tab = tab.clone()
    bad_tab[1, 0] = w.NB + 7
    pa.pa_prefill(out, C.to_dev(q, w.dtype), c.pool, bad_tab, ctx, torch.from_numpy(q_start).cuda(), 300, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & pa.PA_DEV_ERR_BLOCK
    err.zero_()
    bad_ctx = ctx.clone()
    bad_ctx[2] = 100                                     # a 129-token chunk cannot end a 100-token context
    pa.pa_prefill(out, C.to_dev(q, w.dtype), c.pool, tab, bad_ctx, torch.from_numpy(q_start).cuda(), 300, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & pa.PA_DEV_ERR_CTX
    out2, ref, _, _ = _run(c, chunks)
    C.assert_close(out2.cpu().numpy(), ref, "prefill after flagged calls")
