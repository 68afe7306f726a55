"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bit-exact: cache writes, block copies, allocator tables and slots.
Attention outputs (fp32): max |diff| <= 2e-3 and relative L2 <= 1e-3.
Every case, the full-size workloads included, compares every output row.
"""
import os

import numpy as np
import pytest
import torch

import _cases as C
import oracle
import paged_kv_cache_302_gb300 as pa
import workloads as W

pytestmark = pytest.mark.gpu


# ----------------------------------------------------------------------------- cache ops

def test_reshape_and_cache_bit_exact_skips_padding_and_flags_bad_slots():
    w = W.llama3_8b(n_seqs=4)
    rng = np.random.default_rng(1)
    NB, B = 40, 16
    pool = torch.zeros((NB, B, 2, w.H_kv, w.D), dtype=torch.bfloat16, device="cuda")
    host = np.zeros(pool.shape, dtype=np.uint16)
    T = 300
    slots = rng.choice(NB * B, size=T, replace=False).astype(np.int64)
    slots[[5, 17, 200]] = -1
    k, v = W.token_kv(w, T)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache(C.to_dev(k, "bf16"), C.to_dev(v, "bf16"), pool, torch.from_numpy(slots).cuda(),
                            dev_err=err)
    oracle.reshape_and_cache(k, v, host, slots)
    torch.cuda.synchronize()
    assert np.array_equal(C.to_bits(pool), host) and err.item() == 0
    bad = slots.copy()
    bad[3] = NB * B
    before = C.to_bits(pool)
    pa.pa_reshape_and_cache(C.to_dev(k, "bf16"), C.to_dev(v, "bf16"), pool, torch.from_numpy(bad).cuda(),
                            dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & pa.PA_DEV_ERR_SLOT
    assert np.array_equal(C.to_bits(pool), before)   # same data rewritten, bad slot skipped


def test_copy_blocks_bit_exact_and_flags():
    rng = np.random.default_rng(2)
    NB, B, H, D = 30, 16, 8, 128
    bits = W.normal_bits(rng, (NB, B, 2, H, D), "f16")
    pool = C.to_dev(bits, "f16").clone()
    pairs = np.array([[1, 20], [4, 21], [1, 22], [9, 0]], dtype=np.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(pool, torch.from_numpy(pairs).cuda(), dev_err=err)
    oracle.copy_blocks(bits, pairs)
    torch.cuda.synchronize()
    assert np.array_equal(C.to_bits(pool), bits) and err.item() == 0
    pa.pa_copy_blocks(pool, torch.from_numpy(np.array([[2, 3], [3, 5]], dtype=np.int64)).cuda(), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & pa.PA_DEV_ERR_BLOCK
    err.zero_()
    pa.pa_copy_blocks(pool, torch.from_numpy(np.array([[2, NB]], dtype=np.int64)).cuda(), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & pa.PA_DEV_ERR_BLOCK
    for bad in ([[2, 7], [4, 7]], [[6, 6]]):           # a destination named twice; a block copied onto itself
        err.zero_()
        pa.pa_copy_blocks(pool, torch.from_numpy(np.array(bad, dtype=np.int64)).cuda(), dev_err=err)
        torch.cuda.synchronize()
        assert err.item() & pa.PA_DEV_ERR_BLOCK, bad


def test_copy_blocks_many_pairs_over_a_large_pool():
    """20000 pairs over a pool of 300000 one-kilobyte blocks (the chained-pair check then spans three ranges of
    131072 block ids): bit-exact against the oracle with no flag; chains and repeated destinations in the upper
    ranges are flagged."""
    rng = np.random.default_rng(21)
    NB, B, H, D = 300000, 4, 1, 64
    bits = W.normal_bits(rng, (NB, B, 2, H, D), "f16")
    pool = C.to_dev(bits, "f16").clone()
    ids = rng.permutation(NB)[:40000].astype(np.int64)
    pairs = np.stack([ids[:20000], ids[20000:]], axis=1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(pool, torch.from_numpy(pairs).cuda(), dev_err=err)
    oracle.copy_blocks(bits, pairs)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(C.to_bits(pool), bits)
    for bad in ([[270000, 280000], [280000, 5]], [[3, 299999], [4, 299999]], [[10, 20], [262150, 299000],
                                                                            [299000, 11]]):
        err.zero_()
        pa.pa_copy_blocks(pool, torch.from_numpy(np.array(bad, dtype=np.int64)).cuda(), dev_err=err)
        torch.cuda.synchronize()
        assert err.item() & pa.PA_DEV_ERR_BLOCK, bad


def test_table_updates_keep_the_device_tables_current():
    """Device tables patched with the allocator's updates equal freshly packed host tables, bit for bit."""
    w = W.cow(prompts=4, samples=8)
    a = pa.BlockAllocator(w.NB, w.B, w.free_order)
    for p in range(w.prompts):
        a.add_seq(p * w.samples)
        a.append_slots(p * w.samples, w.prompt_len)
        for j in range(1, w.samples):
            a.fork(p * w.samples, p * w.samples + j)
    order = list(np.random.default_rng(5).permutation(w.N))   # device rows in an arbitrary sequence order
    MB = w.max_blocks_per_seq(grow=64)
    tab0, _ = a.block_tables(order, MB)
    dev = torch.from_numpy(tab0).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(6)
    for step in range(6):
        n_tok = rng.integers(0, 40, size=w.N).astype(np.int32)     # first step: copy-on-write for 7 of 8 samples
        _, pairs, upd = a.append_batch(order, n_tok, table_updates=True)
        if step == 0:
            assert len(pairs) > 0
        pa.pa_update_block_tables(dev, torch.from_numpy(np.ascontiguousarray(upd)).cuda(), dev_err=err)
        want, _ = a.block_tables(order, MB)
        torch.cuda.synchronize()
        assert np.array_equal(dev.cpu().numpy(), want) and err.item() == 0
    pad = torch.tensor([[-1, 0, 1], [-7, MB + 3, 2]], dtype=torch.int32, device="cuda")  # padding rows
    pa.pa_update_block_tables(dev, pad, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0 and np.array_equal(dev.cpu().numpy(), want)
    bad = torch.tensor([[w.N, 0, 1], [0, MB, 1]], dtype=torch.int32, device="cuda")
    pa.pa_update_block_tables(dev, bad, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & pa.PA_DEV_ERR_BLOCK
    assert np.array_equal(dev.cpu().numpy(), want)


# ----------------------------------------------------------------------------- decode, every output

def test_tiny_worked_example_every_output():
    w = W.tiny()
    c = C.build_paged(w)
    assert list(c.tables[0][:2]) == [7, 1] and list(c.tables[1][:2]) == [3, 5]
    ref = C.oracle_decode(c)
    for pt in (0, -1, 32):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = C.gpu_decode(c, partition_tokens=pt, dev_err=err).cpu().numpy()
        C.assert_close(out, ref, f"tiny pt={pt}")
        assert err.item() == 0


@pytest.mark.parametrize("pt", [0, -1, 32, 96])
def test_llama_shaped_small_every_output(pt):
    w = W.llama3_8b(n_seqs=24)
    c = C.build_paged(w)
    ref = C.oracle_decode(c)
    out = C.gpu_decode(c, partition_tokens=pt).cpu().numpy()
    C.assert_close(out, ref, f"llama small pt={pt}")


def test_opt13b_shaped_small_every_output():
    w = W.opt13b(n_seqs=6)
    c = C.build_paged(w)
    ref = C.oracle_decode(c)
    out = C.gpu_decode(c).cpu().numpy()
    C.assert_close(out, ref, "opt13b small")


@pytest.mark.parametrize("B", [8, 16, 32])
def test_yi34b_shaped_block_sizes_every_output(B):
    w = W.yi34b_long(n_seqs=2, ctx_len=1500 + B, B=B)
    c = C.build_paged(w)
    ref = C.oracle_decode(c)
    for pt in (0, -1):
        out = C.gpu_decode(c, partition_tokens=pt).cpu().numpy()
        C.assert_close(out, ref, f"yi34b B={B} pt={pt}")


def test_ragged_lengths_cover_every_tail():
    # contexts 1..70 exercise empty / partial 16-token tiles and partial stages
    base = W.llama3_8b(n_seqs=70)
    base.ctx = np.arange(1, 71, dtype=np.int32)
    c = C.build_paged(base)
    ref = C.oracle_decode(c)
    for pt in (-1, 32):
        out = C.gpu_decode(c, partition_tokens=pt).cpu().numpy()
        C.assert_close(out, ref, f"ragged pt={pt}")


def test_single_token_contexts_return_that_token_value_row():
    """Degenerate case: with ctx = 1 the softmax weight is 1, so every head returns V_0 (to within the fp32
    rounding of the base-2 exponent of a product's residual: a relative 4e-7)."""
    N, NB = 300, 400
    w = W.Workload("ctx1", 21, N, 32, 8, 128, 16, "bf16", np.ones(N, np.int32), NB,
                   np.random.default_rng(21).permutation(NB).astype(np.int32))
    c = C.build_paged(w)
    out = C.gpu_decode(c).cpu().numpy()
    v0 = W.bits_to_float(c.host_pool[c.tables[:, 0], 0, 1], w.dtype)          # [N, H_kv, D]
    want = np.repeat(v0, w.G, axis=1).astype(np.float32)                         # head h reads KV head h // G
    np.testing.assert_allclose(out, want, rtol=4e-7, atol=0)


def test_many_short_sequences_every_output():
    """5000 sequences of 1..40 tokens: the schedule handles several sequences per thread, most work items are
    single ragged partitions, and every output is checked."""
    rng = np.random.default_rng(22)
    N, B = 5000, 16
    ctx = rng.integers(1, 41, size=N).astype(np.int32)
    NB = int(((ctx + B - 1) // B).sum()) + 16
    w = W.Workload("many", 22, N, 8, 2, 64, B, "f16", ctx, NB, rng.permutation(NB).astype(np.int32))
    c = C.build_paged(w)
    ref = C.oracle_decode(c)
    for pt in (0, 32):
        C.assert_close(C.gpu_decode(c, partition_tokens=pt).cpu().numpy(), ref, f"many short pt={pt}")


def _schedule_view(ws, N, maxrec):
    """(records [n, 4] int32 rows (seq, kv head, partition, ctx), per-sequence partition counts) that a decode call
    left in its workspace.  White box: the workspace holds a 16-byte header (record count in word 0), the
    per-sequence partition counts and the records, each part starting on a 256-byte boundary."""
    off = (256 + 4 * N + 255) // 256 * 256
    b = ws[: off + 16 * maxrec].cpu().numpy()
    total = int(b[:4].view(np.int32)[0])
    assert 0 <= total <= maxrec
    return b[off: off + 16 * total].view(np.int32).reshape(total, 4), b[256: 256 + 4 * N].view(np.int32).copy()


def _default_partition() -> int:
    """The partition length partition_tokens=0 stands for: 512, or PA_DECODE_PARTITION when that names a positive
    multiple of the 32-token stage (the library reads the variable once per process)."""
    v = os.environ.get("PA_DECODE_PARTITION", "")
    x = int(v) if v.strip().lstrip("-").isdigit() else 0
    return x if x > 0 and x % 32 == 0 else 512


@pytest.mark.parametrize("N,H_kv,pt,max_len", [(1, 8, 0, 3000), (33, 8, 0, 3000), (256, 8, 0, 8192),
                                                 (5000, 2, 64, 200), (40000, 1, -1, 700), (200000, 1, 32, 60)],
                         ids=["1", "33", "256", "5000-pt64", "40000-whole", "200000-pt32"])
def test_schedule_covers_every_work_item_once_longest_first(N, H_kv, pt, max_len):
    """The schedule's work records, read back from a poisoned workspace: exactly one per (sequence, kv head,
    partition); the whole partitions first, in (sequence, partition, kv head) order; then each ragged last
    partition as H_kv consecutive records, by non-increasing length in bins of one 32-token stage.  The batches
    run from one CTA to one per SM, with slices above 1024 sequences at the largest size.  Sampled outputs match
    the oracle (the tables point into a small shared pool, so sequences share blocks)."""
    rng = np.random.default_rng(N)
    B, D, H_q, NB = 16, 64, 2 * H_kv, 64
    PT = {0: _default_partition(), -1: 1 << 30}.get(pt, pt)
    ctx = rng.integers(1, max_len + 1, size=N).astype(np.int32)
    ctx[0] = max_len
    MB = (max_len + B - 1) // B
    tables = rng.integers(0, NB, size=(N, MB)).astype(np.int32)
    pool_bits = W.normal_bits(rng, (NB, B, 2, H_kv, D), "f16")
    q_bits = W.normal_bits(rng, (N, H_q, D), "f16")
    ws = torch.full((pa.pa_decode_workspace_bytes(N, H_q, H_kv, D, max_len, pt),), 0xAB, dtype=torch.uint8,
                    device="cuda")
    out = torch.empty((N, H_q, D), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode(out, C.to_dev(q_bits, "f16"), C.to_dev(pool_bits, "f16"), torch.from_numpy(tables).cuda(),
                 torch.from_numpy(ctx).cuda(), max_len, partition_tokens=pt, workspace=ws, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    P = (ctx.astype(np.int64) + PT - 1) // PT
    rec, nparts = _schedule_view(ws, N, int(P.sum()) * H_kv)
    assert np.array_equal(nparts, P)
    s, h, p, c = (x.astype(np.int64) for x in rec.T)
    assert rec.shape[0] == P.sum() * H_kv
    assert np.array_equal(c, ctx[s])
    keys = np.sort((s * H_kv + h) * P.max() + p)
    seq = np.repeat(np.arange(N), P * H_kv)
    part = np.concatenate([np.repeat(np.arange(n), H_kv) for n in P])
    want = np.sort((seq * H_kv + np.tile(np.arange(H_kv), int(P.sum()))) * P.max() + part)
    assert np.array_equal(keys, want), "some work item is missing or repeated"
    nf = ctx.astype(np.int64) // PT
    F = int(nf.sum()) * H_kv
    whole = (p + 1) * PT <= c
    assert whole[:F].all() and not whole[F:].any()
    ws_seq = np.repeat(np.arange(N), nf * H_kv)
    ws_part = np.concatenate([np.repeat(np.arange(n), H_kv) for n in nf]) if F else np.zeros(0, np.int64)
    assert np.array_equal(s[:F], ws_seq) and np.array_equal(p[:F], ws_part)
    assert np.array_equal(h[:F], np.tile(np.arange(H_kv), F // H_kv))
    ts, th = s[F:].reshape(-1, H_kv), h[F:].reshape(-1, H_kv)
    assert (ts == ts[:, :1]).all() and (th == np.arange(H_kv)).all()
    bins = (c[F:] - p[F:] * PT + 31) // 32
    assert np.all(np.diff(bins) <= 0), "ragged partitions out of longest-first order"
    pick = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, size=22)]))
    pairs = np.array([(x, y) for x in pick for y in (0, H_q - 1)], dtype=np.int32)
    ref = oracle.paged_decode(q_bits, pool_bits, tables, ctx, "f16", pairs=pairs)
    got = out.cpu().numpy()
    C.assert_close(got[pairs[:, 0], pairs[:, 1]], ref[pairs[:, 0], pairs[:, 1]], f"schedule N={N}")


def test_decode_right_after_a_cache_write_reads_the_new_token():
    """A decode launched right after the cache write on the same stream, with no synchronisation between them,
    reads the token the write just stored, also where that token completes a whole 512-token partition (the
    attention kernel streams its first whole partition while the schedule is still being written).  The new
    token's key is aligned with its queries, so it dominates every row's softmax: a stale read would show."""
    rng = np.random.default_rng(31)
    N, B = 48, 16
    ctx = rng.choice([512, 1024, 1536, 2048, 700, 1500], size=N).astype(np.int32)
    ctx[:6] = [512, 1024, 1536, 2048, 2560, 3072]
    NB = int(((ctx + B - 1) // B).sum()) + 16
    w = W.Workload("after_write", 31, N, 32, 8, 128, B, "bf16", ctx, NB, rng.permutation(NB).astype(np.int32))
    c = C.build_paged(w, check_pool=False)
    tab, ctx = c.dev_tables()
    last = c.ctx - 1
    slots = (c.tables[np.arange(w.N), last // w.B].astype(np.int64) * w.B + last % w.B)
    q = W.bits_to_float(c.q, w.dtype).reshape(w.N, w.H_kv, w.G, w.D)
    for it in range(4):
        k_new = W.round_bits(4.0 * q[:, :, it % w.G, :], w.dtype)                     # [N, H_kv, D]
        v_new = W.normal_bits(rng, (w.N, w.H_kv, w.D), w.dtype)
        oracle.reshape_and_cache(k_new, v_new, c.host_pool, slots)
        qd = C.to_dev(c.q, w.dtype)
        kd, vd, sd = C.to_dev(k_new, w.dtype), C.to_dev(v_new, w.dtype), torch.from_numpy(slots).cuda()
        out = torch.full((w.N, w.H_q, w.D), float("nan"), device="cuda")
        torch.cuda.synchronize()
        pa.pa_reshape_and_cache(kd, vd, c.pool, sd)
        pa.pa_decode(out, qd, c.pool, tab, ctx, int(c.ctx.max()))
        torch.cuda.synchronize()
        C.assert_close(out.cpu().numpy(), C.oracle_decode(c), f"decode after write, round {it}")


_GUARD = 4096  # bytes of sentinel before and after a carved buffer (keeps 32-byte alignment)


def _carved(shape, dtype):
    """(backing buffer, tensor of `shape`) with the tensor carved out of the middle of a device buffer whose
    first and last _GUARD bytes hold the sentinel 0x5A."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    big = torch.full((2 * _GUARD + n,), 0x5A, dtype=torch.uint8, device="cuda")
    return big, big[_GUARD: _GUARD + n].view(dtype).view(shape)


def _margins_intact(*bigs):
    torch.cuda.synchronize()
    for big in bigs:
        edge = torch.cat([big[:_GUARD], big[-_GUARD:]])
        assert bool((edge == 0x5A).all()), "a kernel wrote outside its buffer"


def test_no_call_writes_outside_its_buffers():
    """Every device buffer of the tiny worked example (pool, slots, tables, query, output, workspace, copy pairs,
    table updates) and of a small prefill is carved out of a larger allocation with sentinel margins; after
    cache writes, block copies, table updates, decodes in all partition modes and a prefill, the margins are
    unchanged, and the results still match the oracle."""
    w = W.tiny()
    alloc = pa.BlockAllocator(w.NB, w.B, w.free_order)
    slots = []
    for sq in range(w.N):
        alloc.add_seq(sq)
        slots.append(alloc.append_slots(sq, int(w.ctx[sq]))[0])
    slots = np.concatenate(slots)
    tables, ctx = alloc.block_tables(list(range(w.N)), w.max_blocks_per_seq())
    k, v = W.token_kv(w, slots.size)
    shape = (w.NB, w.B, 2, w.H_kv, w.D)
    pool_big, pool = _carved(shape, torch.float16)
    pool.view(torch.int16).fill_(C.nan16(w.dtype))
    host = np.full(shape, W.NAN_BITS[w.dtype], dtype=np.uint16)
    bigs = [pool_big]

    def dev(a, dtype):
        big, t = _carved(a.shape, dtype)
        t.copy_(torch.from_numpy(np.ascontiguousarray(a)).view(dtype) if dtype in (torch.float16, torch.bfloat16)
                else torch.from_numpy(np.ascontiguousarray(a)))
        bigs.append(big)
        return t

    kd, vd = dev(k.view(np.int16), torch.float16), dev(v.view(np.int16), torch.float16)
    pa.pa_reshape_and_cache(kd, vd, pool, dev(slots, torch.int64))
    oracle.reshape_and_cache(k, v, host, slots)
    free = sorted(set(range(w.NB)) - set(tables[tables >= 0].tolist()))
    pairs = np.array([[tables[3][0], free[0]], [tables[2][1], free[1]]], dtype=np.int64)
    pa.pa_copy_blocks(pool, dev(pairs, torch.int64))
    oracle.copy_blocks(host, pairs)
    _margins_intact(*bigs)
    assert np.array_equal(C.to_bits(pool), host)
    tab, ctx_d = dev(tables, torch.int32), dev(ctx.astype(np.int32), torch.int32)
    q = W.queries(w)
    qd = dev(q.view(np.int16), torch.float16)
    ref = oracle.paged_decode(q, host, tables, ctx, w.dtype)
    for pt in (0, -1, 32):
        out_big, out = _carved((w.N, w.H_q, w.D), torch.float32)
        ws_big, ws = _carved((pa.pa_decode_workspace_bytes(w.N, w.H_q, w.H_kv, w.D, int(ctx.max()), pt),), torch.uint8)
        ws.fill_(0xAB)
        pa.pa_decode(out, qd, pool, tab, ctx_d, int(ctx.max()), partition_tokens=pt, workspace=ws)
        _margins_intact(out_big, ws_big, *bigs)
        C.assert_close(out.cpu().numpy(), ref, f"guarded decode pt={pt}")
    upd = np.array([[0, 1, free[2]], [3, 2, free[3]], [-1, 0, 0]], dtype=np.int32)
    pa.pa_update_block_tables(tab, dev(upd, torch.int32))
    _margins_intact(*bigs)
    want = tables.copy()
    want[0, 1], want[3, 2] = free[2], free[3]
    assert np.array_equal(tab.cpu().numpy(), want)

    # prefill (blocks of 16 tokens): chunks of the last 40 and 100 tokens of two short sequences
    ctx_p = np.array([300, 130], dtype=np.int32)
    NBp = int(((ctx_p + 15) // 16).sum()) + 8
    wp = W.Workload("guard_prefill", 4, 2, 32, 8, 128, 16, "bf16", ctx_p, NBp,
                    np.random.default_rng(4).permutation(NBp).astype(np.int32))
    cp = C.build_paged(wp)
    chunks = [40, 100]
    q_start = np.array([0, 40, 140], dtype=np.int32)
    qp = W.normal_bits(np.random.default_rng(4), (140, wp.H_q, wp.D), wp.dtype)
    out_big, outp = _carved((140, wp.H_q, wp.D), torch.float32)
    pt_tab, pt_ctx = cp.dev_tables()
    qs_big, qs_d = _carved((3,), torch.int32)
    qs_d.copy_(torch.from_numpy(q_start))
    q_big, q_d = _carved(qp.shape, torch.bfloat16)
    q_d.copy_(torch.from_numpy(qp.view(np.int16)).view(torch.bfloat16))
    pws_big, pws = _carved((pa.pa_prefill_workspace_bytes(wp.N, wp.H_kv, wp.D, wp.B, cp.MB),), torch.uint8)
    refp = oracle.paged_prefill(qp, cp.host_pool, cp.tables, cp.ctx, q_start, wp.dtype, nthreads=0)
    for stage_v in (True, False):            # V staged as fp16 in the workspace, and P split without one
        pa.pa_prefill(outp, q_d, cp.pool, pt_tab, pt_ctx, qs_d, max(chunks), workspace=pws, stage_v=stage_v)
        _margins_intact(out_big, qs_big, q_big, pws_big)
        C.assert_close(outp.cpu().numpy(), refp, f"guarded prefill, stage_v={stage_v}")


def test_block_relabelling_gives_identical_bits():
    w = W.llama3_8b(n_seqs=12)
    c = C.build_paged(w, check_pool=False)
    out1 = C.gpu_decode(c).cpu()
    perm = np.random.default_rng(3).permutation(w.NB)
    pool2 = torch.empty_like(c.pool)
    pool2[torch.from_numpy(perm).cuda()] = c.pool
    tables2 = np.where(c.tables >= 0, perm[np.maximum(c.tables, 0)], -1).astype(np.int32)
    c2 = C.Paged(w, pool2, None, tables2, c.ctx, c.q)
    out2 = C.gpu_decode(c2).cpu()
    assert torch.equal(out1, out2)


def test_contiguous_layout_matches_paged_bit_for_bit_and_oracle():
    w = W.yi34b_long(n_seqs=3, ctx_len=2000, B=16)
    w.ctx = np.array([2000, 1333, 77], dtype=np.int32)
    c = C.build_paged(w)
    N_max, S_max = 5, 2048
    req = np.array([3, 0, 4], dtype=np.int32)
    kb = torch.zeros((N_max, S_max, w.H_kv, w.D), dtype=torch.bfloat16, device="cuda")
    vb = torch.zeros_like(kb)
    kb.view(torch.int16).fill_(C.nan16("bf16"))
    vb.view(torch.int16).fill_(C.nan16("bf16"))
    hk = np.full(kb.shape, W.NAN_BITS["bf16"], dtype=np.uint16)
    hv = hk.copy()
    for s in range(w.N):
        t = np.arange(int(w.ctx[s]))
        phys = c.tables[s, t // w.B]
        hk[req[s], : len(t)] = c.host_pool[phys, t % w.B, 0]
        hv[req[s], : len(t)] = c.host_pool[phys, t % w.B, 1]
    kb.copy_(C.to_dev(hk, "bf16"))
    vb.copy_(C.to_dev(hv, "bf16"))
    ref = oracle.contiguous_decode(c.q, hk, hv, req, w.ctx, "bf16")
    for pt in (0, -1):
        paged = C.gpu_decode(c, partition_tokens=pt)
        out = torch.full_like(paged, float("nan"))
        pa.pa_decode_contiguous(out, C.to_dev(c.q, "bf16"), kb, vb, torch.from_numpy(req).cuda(),
                                torch.from_numpy(w.ctx).cuda(), int(w.ctx.max()), partition_tokens=pt)
        torch.cuda.synchronize()
        assert torch.equal(out, paged)
        C.assert_close(out.cpu().numpy(), ref, f"contiguous pt={pt}")


@pytest.mark.parametrize("make", [lambda: W.llama3_8b(n_seqs=10), lambda: W.opt13b(n_seqs=6)],
                         ids=["bf16", "fp16"])
def test_low_precision_output_is_the_rounded_fp32_output(make):
    """A 16-bit output = round-to-nearest-even of the fp32 output of the same call, bit for bit, and within the
    fp32 tolerance plus half an ulp of the oracle: unpartitioned, 512-token partitions (warp-per-row merge) and
    32-token partitions (at least 32 per row: CTA-per-row merge)."""
    w = make()
    c = C.build_paged(w)
    ref = C.oracle_decode(c)
    odt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    assert (int(c.ctx.max()) + 31) // 32 >= 32
    for pt in (0, -1, 32):
        out32 = C.gpu_decode(c, partition_tokens=pt).cpu().numpy()
        out16 = C.gpu_decode(c, partition_tokens=pt, out_dtype=odt)
        bits = C.to_bits(out16)
        assert np.array_equal(bits, W.round_bits(out32, w.dtype))
        half_ulp = np.abs(W.bits_to_float(bits + 1, w.dtype) - W.bits_to_float(bits, w.dtype)) / 2
        assert np.all(np.abs(W.bits_to_float(bits, w.dtype) - ref) <= C.ATOL + half_ulp)


def test_output_in_pinned_host_memory_equals_device_output():
    """out may live in pinned host memory: the attention kernel (single-partition rows) and both merge kernels
    write the rows across the host link, bit for bit what they write into device memory, fp32 and 16-bit."""
    w = W.llama3_8b(n_seqs=10)
    c = C.build_paged(w)
    tab, ctx = c.dev_tables()
    qd = C.to_dev(c.q, w.dtype)
    ref = C.oracle_decode(c)
    for odt in (torch.float32, torch.bfloat16):
        for pt in (0, -1, 32):
            dev_out = torch.full((w.N, w.H_q, w.D), float("nan"), dtype=odt, device="cuda")
            host_out = torch.full((w.N, w.H_q, w.D), float("nan"), dtype=odt).pin_memory()
            pa.pa_decode(dev_out, qd, c.pool, tab, ctx, int(c.ctx.max()), partition_tokens=pt)
            pa.pa_decode(host_out, qd, c.pool, tab, ctx, int(c.ctx.max()), partition_tokens=pt)
            torch.cuda.synchronize()
            assert torch.equal(dev_out.cpu(), host_out), f"{odt} pt={pt}"
            if odt == torch.float32:
                C.assert_close(host_out.numpy(), ref, f"host output pt={pt}")
    with pytest.raises(pa.PAError):
        pa.pa_decode(torch.empty((w.N, w.H_q, w.D)), qd, c.pool, tab, ctx, int(c.ctx.max()))  # pageable: refused


@pytest.mark.parametrize("R,P,D", [(37, 9, 128), (37, 40, 128), (11, 300, 128), (23, 33, 64)])
def test_partition_reduce_standalone_matches_oracle_merge(R, P, D):
    """Warp-per-row merge (P < 32) and CTA-per-row merge (P >= 32, rows of up to 300 partitions)."""
    rng = np.random.default_rng(4 + P)
    m2 = (rng.normal(size=(R, P)) * 3).astype(np.float32)
    l = rng.uniform(0.5, 40.0, size=(R, P)).astype(np.float32)
    acc = rng.normal(size=(R, P, D)).astype(np.float32)
    nparts = rng.integers(1, P + 1, size=R).astype(np.int32)
    ref = oracle.partition_merge(m2.astype(np.float64), l.astype(np.float64), acc.astype(np.float64), nparts)
    out = torch.full((R, D), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_partition_reduce(out, torch.from_numpy(m2).cuda(), torch.from_numpy(l).cuda(),
                           torch.from_numpy(acc).cuda(), torch.from_numpy(nparts).cuda(), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=2e-5, atol=2e-5)


def test_device_errors_are_flagged_not_faulted():
    w = W.llama3_8b(n_seqs=6)
    c = C.build_paged(w)
    tab, ctx = c.dev_tables()
    qd = C.to_dev(c.q, w.dtype)
    out = torch.zeros((w.N, w.H_q, w.D), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_ctx = ctx.clone()
    bad_ctx[2] = 0
    pa.pa_decode(out, qd, c.pool, tab, bad_ctx, int(c.ctx.max()), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & pa.PA_DEV_ERR_CTX
    err.zero_()
    bad_tab = tab.clone()
    bad_tab[1, 0] = w.NB + 5
    pa.pa_decode(out, qd, c.pool, bad_tab, ctx, int(c.ctx.max()), dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & pa.PA_DEV_ERR_BLOCK
    # the context is still usable afterwards
    out2 = C.gpu_decode(c).cpu().numpy()
    C.assert_close(out2, C.oracle_decode(c), "after flagged calls")


# ----------------------------------------------------------------------------- full-size workloads, every row

def _full_check(c, pts=(0,)):
    """Every (sequence, query head) row of a full-size workload against the oracle (all host cores)."""
    ref = C.oracle_decode(c)
    for pt in pts:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = C.gpu_decode(c, partition_tokens=pt, dev_err=err).cpu().numpy()
        assert err.item() == 0
        C.assert_close(out, ref, f"{c.w.name} pt={pt}")
    return ref


def test_full_opt13b():
    _full_check(C.build_paged(W.opt13b()), pts=(0, -1))


def test_full_llama3_8b():
    _full_check(C.build_paged(W.llama3_8b()), pts=(0, -1))


def test_full_cow_parallel_sampling():
    c, npairs = C.build_cow(W.cow())
    assert npairs == 224
    _full_check(c)


@pytest.mark.parametrize("B", [8, 16, 32])
def test_full_yi34b_long_context(B):
    _full_check(C.build_paged(W.yi34b_long(B=B), check_pool=(B == 16)))


def test_full_yi34b_contiguous_layout():
    """The unpaged comparison at its full size: 8 requests x 32768 tokens in per-request K/V buffers
    [N_max, S_max, H_kv, D] at offset reqId * S_max, every row against the oracle's contiguous decode and bit
    for bit against the paged decode of the same K/V."""
    w = W.yi34b_long(B=16)
    c = C.build_paged(w, check_pool=False)
    N_max, S_max = w.N, int(c.ctx.max())
    req = W.request_ids(w, N_max)
    host_k = np.zeros((N_max, S_max, w.H_kv, w.D), dtype=np.uint16)
    host_v = np.zeros_like(host_k)
    for s in range(w.N):
        blocks = c.tables[s, : -(-int(c.ctx[s]) // w.B)]
        rows = c.host_pool[blocks].reshape(-1, 2, w.H_kv, w.D)[: int(c.ctx[s])]
        host_k[req[s], : rows.shape[0]] = rows[:, 0]
        host_v[req[s], : rows.shape[0]] = rows[:, 1]
    kb, vb = C.to_dev(host_k, w.dtype), C.to_dev(host_v, w.dtype)
    tab, ctx = c.dev_tables()
    qd = C.to_dev(c.q, w.dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((w.N, w.H_q, w.D), float("nan"), device="cuda")
    pa.pa_decode_contiguous(out, qd, kb, vb, torch.from_numpy(req).cuda(), ctx, S_max, dev_err=err)
    paged = C.gpu_decode(c)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out, paged), "contiguous and paged outputs differ"
    ref = oracle.contiguous_decode(c.q, host_k, host_v, req, c.ctx, w.dtype, nthreads=0)
    C.assert_close(out.cpu().numpy(), ref, "yi34b contiguous, full size")


# ----------------------------------------------------------------------------- swap and beam search

def test_swap_out_and_back_in_is_bit_exact_and_decodes_identically():
    w = W.llama3_8b(n_seqs=8, grow=8192)        # enough spare blocks to move the longest sequence
    c = C.build_paged(w, check_pool=False)
    rng = np.random.default_rng(8)
    s = int(np.argmax(w.ctx))
    nb = -(-int(w.ctx[s]) // w.B)
    blocks = c.tables[s, :nb].astype(np.int64)
    NBh = nb + 40
    host_pool = torch.zeros((NBh, w.B, 2, w.H_kv, w.D), dtype=torch.bfloat16).pin_memory()
    host_ids = rng.choice(NBh, size=nb, replace=False).astype(np.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_pairs = torch.from_numpy(np.stack([blocks, host_ids], axis=1)).cuda()          # swap out: device -> host
    pa.pa_swap_blocks(host_pool, c.pool, out_pairs, dev_err=err)
    torch.cuda.synchronize()
    dev_bits = C.to_bits(c.pool)
    want = np.zeros(host_pool.shape, dtype=np.uint16)
    oracle.swap_blocks(want, dev_bits, np.stack([blocks, host_ids], axis=1))
    assert np.array_equal(host_pool.view(torch.int16).numpy().view(np.uint16), want) and err.item() == 0
    used = set(c.tables[c.tables >= 0].tolist())
    free = np.array([b for b in range(w.NB) if b not in used][:nb], dtype=np.int64)
    in_pairs = torch.from_numpy(np.stack([host_ids, free], axis=1)).pin_memory()       # swap in: host -> device,
    pa.pa_swap_blocks(c.pool, host_pool, in_pairs, dev_err=err)                        # pairs in pinned memory
    torch.cuda.synchronize()
    oracle.swap_blocks(dev_bits, want, np.stack([host_ids, free], axis=1))
    assert np.array_equal(C.to_bits(c.pool), dev_bits) and err.item() == 0
    ref = C.gpu_decode(c)
    moved = c.tables.copy()
    moved[s, :nb] = free
    got = C.gpu_decode(C.Paged(w, c.pool, None, moved, c.ctx, c.q))
    assert torch.equal(ref, got)
    bad = torch.tensor([[0, NBh]], dtype=torch.int64, device="cuda")
    pa.pa_swap_blocks(host_pool, c.pool, bad, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() & pa.PA_DEV_ERR_BLOCK
    with pytest.raises(pa.PAError):
        pa.pa_swap_blocks(torch.zeros_like(host_pool, device="cpu"), c.pool, out_pairs)   # pageable: refused


def test_beam_search_fork_tree_decode_every_output():
    """Beams forked from beams: copy-on-write pairs copied on the device before the writes, then every
    live beam decoded; pool bit-exact and outputs against the oracle."""
    from oracle.alloc_model import AllocModel
    shape = W.llama3_8b(n_seqs=1)
    NB, B = 256, 16
    order = np.random.default_rng(7).permutation(NB)
    a = pa.BlockAllocator(NB, B, order)
    m = AllocModel(NB, B, order)
    pool = torch.empty((NB, B, 2, shape.H_kv, shape.D), dtype=torch.bfloat16, device="cuda")
    pool.view(torch.int16).fill_(C.nan16("bf16"))
    host = np.full(pool.shape, W.NAN_BITS["bf16"], dtype=np.uint16)
    rng = np.random.default_rng(9)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    live = []
    for op in W.beam_search_ops():
        kind = op[0]
        if kind == "add":
            a.add_seq(op[1]); m.add_seq(op[1])
        elif kind == "fork":
            a.fork(op[1], op[2]); m.fork(op[1], op[2])
        elif kind == "free":
            a.free_seq(op[1]); m.free_seq(op[1])
        elif kind == "append":
            slots, pairs = a.append_slots(op[1], op[2])
            ms, mp = m.append_slots(op[1], op[2])
            assert list(slots) == ms and [tuple(r) for r in pairs] == mp
            if len(mp):
                pa.pa_copy_blocks(pool, torch.from_numpy(np.ascontiguousarray(pairs)).cuda(), dev_err=err)
                oracle.copy_blocks(host, np.asarray(mp, dtype=np.int64))
            k = W.normal_bits(rng, (op[2], shape.H_kv, shape.D), "bf16")
            v = W.normal_bits(rng, (op[2], shape.H_kv, shape.D), "bf16")
            pa.pa_reshape_and_cache(C.to_dev(k, "bf16"), C.to_dev(v, "bf16"), pool, torch.from_numpy(slots).cuda(),
                                    dev_err=err)
            oracle.reshape_and_cache(k, v, host, np.asarray(ms, dtype=np.int64))
        else:
            live = list(op[1])
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(C.to_bits(pool), host)
    MB = 8
    tables, ctx = a.block_tables(live, MB)
    q = W.normal_bits(rng, (len(live), shape.H_q, shape.D), "bf16")
    wl = W.Workload("beams", 0, len(live), shape.H_q, shape.H_kv, shape.D, B, "bf16", ctx, NB, order)
    c = C.Paged(wl, pool, host, tables, ctx, q)
    for pt in (0, -1, 32):
        C.assert_close(C.gpu_decode(c, partition_tokens=pt).cpu().numpy(), C.oracle_decode(c), f"beams pt={pt}")
