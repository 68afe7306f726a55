"""GPU parity of the tcgen05 paged prefill against the fp64 oracle (causal, chunked)."""
import numpy as np
import pytest
import torch

import _cases as C
import oracle
import paged_kv_cache_302_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu


def _run(c, chunks, seed=0, out_dtype=torch.float32, rows=None, stage_v=True):
    w = c.w
    rng = np.random.default_rng(seed)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(q_start[-1])
    q = W.normal_bits(rng, (T, w.H_q, w.D), w.dtype)
    tab, ctx = c.dev_tables()
    out = torch.full((T, w.H_q, w.D), float("nan"), dtype=out_dtype, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_prefill(out, C.to_dev(q, w.dtype), c.pool, tab, ctx, torch.from_numpy(q_start).cuda(), int(max(chunks)),
                  dev_err=err, stage_v=stage_v)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle.paged_prefill(q, c.host_pool, c.tables, c.ctx, q_start, w.dtype, rows=rows, nthreads=0)
    return out, ref, q, q_start


def _with_ctx(w, ctx):
    w.ctx = np.asarray(ctx, dtype=np.int32)
    return w


def _kernel(monkeypatch, kernel):
    """Selects the prefill kernel of the call: "wide" (the default: persistent 2-CTA clusters, one query tile per
    CTA, 256-key tiles, for fp16 caches and staged bf16 rows) or "narrow" (two query tiles per CTA, 128-key tiles,
    for every row)."""
    monkeypatch.setenv("PA_PREFILL_KERNEL", kernel)


@pytest.mark.parametrize("kernel", ["wide", "narrow"])
@pytest.mark.parametrize("stage_v", [True, False], ids=["staged_v", "split_p"])
@pytest.mark.parametrize("chunks_of", ["full", "tail", "mixed"])
def test_prefill_llama_shaped_every_output(chunks_of, stage_v, kernel, monkeypatch):
    _kernel(monkeypatch, kernel)
    w = _with_ctx(W.llama3_8b(n_seqs=4), [200, 513, 77, 1000])
    c = C.build_paged(w)
    chunks = {"full": list(w.ctx), "tail": [1, 1, 1, 1], "mixed": [200, 130, 1, 257]}[chunks_of]
    out, ref, _, _ = _run(c, chunks, stage_v=stage_v)
    C.assert_close(out.cpu().numpy(), ref, f"prefill {chunks_of}")


@pytest.mark.parametrize("stage_v", [True, False], ids=["staged_v", "split_p"])
@pytest.mark.parametrize("make,ctx,chunks", [
    (lambda: W.opt13b(n_seqs=3), [300, 129, 700], [300, 50, 129]),         # MHA, fp16
    (lambda: W.yi34b_long(n_seqs=2, ctx_len=600, B=8), [600, 331], [600, 200]),   # G = 7, B = 8
    (lambda: W.yi34b_long(n_seqs=2, ctx_len=600, B=32), [600, 331], [333, 331]),  # B = 32
])
@pytest.mark.parametrize("kernel", ["wide", "narrow"])
def test_prefill_group_sizes_and_block_sizes(make, ctx, chunks, stage_v, kernel, monkeypatch):
    _kernel(monkeypatch, kernel)
    c = C.build_paged(_with_ctx(make(), ctx))
    out, ref, _, _ = _run(c, chunks, stage_v=stage_v)
    C.assert_close(out.cpu().numpy(), ref, f"prefill {c.w.name}")


@pytest.mark.parametrize("kernel", ["wide", "narrow"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_head_dim_64(dtype, kernel, monkeypatch):
    _kernel(monkeypatch, kernel)
    w = W.Workload("d64", 1, 3, 8, 2, 64, 8, dtype, np.array([100, 9, 256], np.int32), 200,
                   np.random.default_rng(3).permutation(200).astype(np.int32))
    c = C.build_paged(w)
    out, ref, _, _ = _run(c, [100, 9, 129])
    C.assert_close(out.cpu().numpy(), ref, f"prefill D=64 {dtype}")


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


def _scale_v_bits(bits: np.ndarray, log2_factor: int) -> np.ndarray:
    """bf16 bit patterns times 2^log2_factor (exact: only the exponent moves; zeros stay zero)."""
    f = (bits.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** log2_factor)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def test_prefill_workspace_too_small_is_refused():
    w = _with_ctx(W.llama3_8b(n_seqs=2), [300, 129])
    c = C.build_paged(w)
    tab, ctx = c.dev_tables()
    need = pa.pa_prefill_workspace_bytes(w.N, w.H_kv, w.D, w.B, c.MB)
    q = torch.zeros((300, w.H_q, w.D), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((300, w.H_q, w.D), device="cuda")
    qs = torch.tensor([0, 200, 300], dtype=torch.int32, device="cuda")
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    launches = pa.launch_count()
    with pytest.raises(pa.PAError, match="workspace too small"):
        pa.pa_prefill(out, q, c.pool, tab, ctx, qs, 200, workspace=small)
    assert pa.launch_count() == launches


@pytest.mark.parametrize("stage_v", [True, False], ids=["staged_v", "split_p"])
@pytest.mark.parametrize("B", [8, 16])
def test_prefill_bf16_value_groups_outside_the_fp16_range(B, stage_v):
    """bf16 V is staged as fp16 for the value product only where that is exact; a (sequence, KV head) with a V
    magnitude >= 65536 (fp16 would overflow), or with a 32-key group whose values are all below 2^-10 (fp16
    subnormals would drop bits), is computed from the pool with the split P instead.  Sequence 0: every V times
    2^17; sequence 1: every V times 2^-20; sequence 2: one block of V times 2^17 among ordinary ones; sequence 3
    ordinary (staged).  Each output row is checked against the oracle relative to its own magnitude."""
    w = _with_ctx(W.yi34b_long(n_seqs=4, ctx_len=700, B=B), [700, 450, 600, 300])
    c = C.build_paged(w)
    host = c.host_pool
    for s, (blocks, k) in enumerate([(None, 17), (None, -20), ([5], 17)]):
        nb = -(-int(c.ctx[s]) // w.B)
        ids = c.tables[s, :nb] if blocks is None else c.tables[s, blocks]
        for b in ids:
            host[b, :, 1] = _scale_v_bits(host[b, :, 1], k)
    # unused slots of the last blocks were NaN-poisoned and scaled as NaN: NaN stays NaN
    c.pool.copy_(C.to_dev(host, w.dtype).view(c.pool.shape))
    chunks = [700, 300, 600, 300]
    out, ref, _, q_start = _run(c, chunks, stage_v=stage_v)
    got = out.cpu().numpy()
    assert np.all(np.isfinite(got))
    for s in range(w.N):
        g = got[q_start[s]:q_start[s + 1]].reshape(-1, w.D)
        r = ref[q_start[s]:q_start[s + 1]].reshape(-1, w.D)
        scale = np.maximum(np.abs(r).max(axis=1, keepdims=True), 1.0 if s != 1 else 1e-30)
        d = np.abs(g - r) / scale
        assert d.max() <= C.ATOL, f"seq {s}: max row-relative |diff| {d.max():.3e}"
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        assert rel <= C.REL_L2, f"seq {s}: rel L2 {rel:.3e}"


@pytest.mark.parametrize("H_q,H_kv", [(24, 12), (7, 1)], ids=["12_kv_heads", "1_kv_head"])
def test_prefill_bf16_staging_head_groups(H_q, H_kv):
    """V staging takes up to 8 KV heads per CTA: with 12 the second group holds 4 (its TMA box reaches past the
    last head and reads zeros there, which are not written), with 1 a group is one head.  Staged and split
    outputs both against the oracle."""
    ctx = np.array([700, 129, 333], dtype=np.int32)
    NB = int(sum(-(-ctx // 16))) + 32
    w = W.Workload(f"heads{H_kv}", 11, 3, H_q, H_kv, 128, 16, "bf16", ctx, NB,
                   np.random.default_rng(11).permutation(NB).astype(np.int32))
    c = C.build_paged(w)
    for stage_v in (True, False):
        out, ref, _, _ = _run(c, [700, 100, 333], stage_v=stage_v)
        C.assert_close(out.cpu().numpy(), ref, f"prefill H_kv={H_kv} stage_v={stage_v}")


@pytest.mark.parametrize("kernel", ["wide", "narrow"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("G", [16, 40, 128])
def test_prefill_large_head_groups(G, dtype, kernel, monkeypatch):
    """Many query heads per KV head: a 128-row query tile holds 128/G tokens (8, 3 and 1; with G = 40 eight rows
    of each tile are unused), so a chunk spans many query tiles and pairs of them.  Every output against the
    oracle, each prefill kernel in turn."""
    _kernel(monkeypatch, kernel)
    H_kv = 2 if G < 128 else 1
    ctx = np.array([300, 45], dtype=np.int32)
    NB = int(sum(-(-ctx // 16))) + 8
    w = W.Workload(f"group{G}", 21, 2, G * H_kv, H_kv, 128, 16, dtype, ctx, NB,
                   np.random.default_rng(21).permutation(NB).astype(np.int32))
    c = C.build_paged(w)
    out, ref, _, _ = _run(c, [300, 7])
    C.assert_close(out.cpu().numpy(), ref, f"prefill G={G} {dtype} {kernel}")


@pytest.mark.parametrize("kernel", ["wide", "narrow"])
def test_prefill_empty_chunks_and_a_generous_max_q_len(kernel, monkeypatch):
    """Sequences with no chunk rows between others, and max_q_len well above the longest chunk: the units past every
    chunk are empty and write nothing; every row of the chunks against the oracle, and no row outside them is
    touched (the output starts as NaN)."""
    _kernel(monkeypatch, kernel)
    w = _with_ctx(W.llama3_8b(n_seqs=4), [300, 77, 129, 513])
    c = C.build_paged(w)
    chunks = [0, 77, 0, 300]
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(q_start[-1])
    q = W.normal_bits(np.random.default_rng(4), (T, w.H_q, w.D), w.dtype)
    tab, ctx = c.dev_tables()
    out = torch.full((T + 8, w.H_q, w.D), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_prefill(out[:T], C.to_dev(q, w.dtype), c.pool, tab, ctx, torch.from_numpy(q_start).cuda(), 1000, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle.paged_prefill(q, c.host_pool, c.tables, c.ctx, q_start, w.dtype, nthreads=0)
    C.assert_close(out[:T].cpu().numpy(), ref, f"prefill empty chunks {kernel}")
    assert torch.isnan(out[T:]).all(), "rows past the chunks were written"


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_repeated_calls_are_bit_identical(dtype):
    """The persistent 2-CTA kernel's copies, shared free barriers and exit ordering, exercised 200 times back to
    back: every call bit-identical to the first, no device flags.  Chunks of 1000, 37 and 7 tokens give rows with
    an odd number of query tiles (a pair whose second CTA has no rows) and rows far shorter than the longest."""
    w = _with_ctx(W.llama3_8b(n_seqs=3), [1500, 300, 7])
    if dtype == "f16":
        w.dtype = "f16"
    c = C.build_paged(w)
    chunks = [1000, 37, 7]
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(q_start[-1])
    q = C.to_dev(W.normal_bits(np.random.default_rng(9), (T, w.H_q, w.D), w.dtype), w.dtype)
    tab, ctx = c.dev_tables()
    qs = torch.from_numpy(q_start).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = torch.full((T, w.H_q, w.D), float("nan"), device="cuda")
    pa.pa_prefill(first, q, c.pool, tab, ctx, qs, max(chunks), dev_err=err)
    outs = [torch.full_like(first, float("nan")) for _ in range(4)]
    same = torch.ones(1, dtype=torch.bool, device="cuda")
    for i in range(200):
        o = outs[i % 4]
        pa.pa_prefill(o, q, c.pool, tab, ctx, qs, max(chunks), dev_err=err)
        same &= (o == first).all()  # on the device: no synchronisation inside the loop
    torch.cuda.synchronize()
    assert err.item() == 0
    assert bool(same.item()), "a repeated prefill differs from the first call"
    assert np.all(np.isfinite(first.cpu().numpy()))
