"""Pins for the fp64 oracle against values and identities fixed outside it.

Each test ties one oracle function to something other than the oracle itself:
printed numbers from the pages (tests/golden/), library routines (numpy's
binary16 conversion, torch's scaled_dot_product_attention in fp64, scipy's
expit / logsumexp), closed forms, and invariants.  No GPU is involved.
"""
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- 16-bit decoding

def test_half_decoding_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decoding_matches_binary32_upper_half():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ----------------------------------------------------------------------------- size formulas

def _golden_rows(name, kind):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            parts = line.split()
            if parts and parts[0] == kind:
                rows.append(parts[1:])
    return rows


def test_kv_size_formula_reproduces_printed_opt13b_figures():
    rows = _golden_rows("kv_sizes.txt", "kv")
    assert len(rows) == 2
    for name, t, L, H, Dh, expect, tol in rows:
        got = oracle.kv_cache_bytes(float(t), float(L), float(H), float(Dh), 2.0)
        assert abs(got - float(expect)) / float(expect) <= float(tol), name
    # the formula is exactly 4*t*L*H*D_h for fp16
    assert oracle.kv_cache_bytes(1, 40, 40, 128, 2) == 819200.0


def test_tokens_per_page_reproduces_printed_table():
    rows = _golden_rows("kv_sizes.txt", "page")
    assert len(rows) == 4
    for name, page, hkv, d, eb, expect in rows:
        assert oracle.tokens_per_page(float(page), float(hkv), float(d), float(eb)) == float(expect), name


# ----------------------------------------------------------------------------- helpers

def _tiny_paged(rng, N=3, H_q=4, H_kv=2, D=16, B=4, NB=40, dtype="bf16", ctx=(1, 9, 14), poison=True):
    """Random pool with a seeded block assignment; returns q, pool, tables, ctx."""
    ctx = np.array(ctx, dtype=np.int32)
    MB = int(-(-ctx.max() // B))
    order = rng.permutation(NB)
    tables = np.full((N, MB), -1, dtype=np.int32)
    used = 0
    for s in range(N):
        nb = -(-int(ctx[s]) // B)
        tables[s, :nb] = order[used:used + nb]
        used += nb
    pool = W.normal_bits(rng, (NB, B, 2, H_kv, D), dtype)
    if poison:
        nan = W.NAN_BITS[dtype]
        live = np.zeros((NB, B), dtype=bool)
        for s in range(N):
            for t in range(int(ctx[s])):
                live[tables[s, t // B], t % B] = True
        pool[~live] = nan
    q = W.normal_bits(rng, (N, H_q, D), dtype)
    return q, pool, tables, ctx


def _gather_contiguous(pool, tables, ctx):
    """K and V of each sequence in logical order via numpy indexing: [N, S_max, H_kv, D] each."""
    NB, B, _, H_kv, D = pool.shape
    N = len(ctx)
    S = int(ctx.max())
    kb = np.zeros((N, S, H_kv, D), dtype=np.uint16)
    vb = np.zeros((N, S, H_kv, D), dtype=np.uint16)
    for s in range(N):
        t = np.arange(int(ctx[s]))
        phys = tables[s, t // B]
        kb[s, : len(t)] = pool[phys, t % B, 0]
        vb[s, : len(t)] = pool[phys, t % B, 1]
    return kb, vb


def _sdpa_reference(q, kb, vb, ctx, dtype):
    """torch.nn.functional.scaled_dot_product_attention in fp64, one query per sequence, GQA by repetition."""
    qf = torch.from_numpy(W.bits_to_float(q, dtype).astype(np.float64))
    kf = torch.from_numpy(W.bits_to_float(kb, dtype).astype(np.float64))
    vf = torch.from_numpy(W.bits_to_float(vb, dtype).astype(np.float64))
    N, H_q, D = q.shape
    G = H_q // kb.shape[2]
    out = np.zeros((N, H_q, D))
    for s in range(N):
        n = int(ctx[s])
        k = kf[s, :n].permute(1, 0, 2).repeat_interleave(G, dim=0)   # [H_q, n, D]
        v = vf[s, :n].permute(1, 0, 2).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qf[s][:, None, :], k, v)
        out[s] = o[:, 0, :].numpy()
    return out


# ----------------------------------------------------------------------------- attention pins

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_paged_decode_matches_library_attention(dtype):
    rng = np.random.default_rng(11)
    q, pool, tables, ctx = _tiny_paged(rng, N=4, H_q=6, H_kv=2, D=32, B=4, NB=64, dtype=dtype, ctx=(1, 5, 16, 37))
    got = oracle.paged_decode(q, pool, tables, ctx, dtype)
    kb, vb = _gather_contiguous(pool, tables, ctx)
    ref = _sdpa_reference(q, kb, vb, ctx, dtype)
    assert np.all(np.isfinite(got))
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_contiguous_decode_matches_library_attention_with_request_offsets():
    rng = np.random.default_rng(12)
    q, pool, tables, ctx = _tiny_paged(rng, N=3, H_q=4, H_kv=4, D=16, B=8, NB=32, ctx=(3, 20, 11))
    kb, vb = _gather_contiguous(pool, tables, ctx)
    # scatter the requests into a larger buffer at permuted request slots
    req = np.array([4, 0, 2], dtype=np.int32)
    S = kb.shape[1]
    K = W.normal_bits(rng, (5, S + 3, 4, 16), "bf16")
    V = W.normal_bits(rng, (5, S + 3, 4, 16), "bf16")
    K[req, :S] = kb
    V[req, :S] = vb
    got = oracle.contiguous_decode(q, K, V, req, ctx, "bf16")
    ref = _sdpa_reference(q, kb, vb, ctx, "bf16")
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # paged and contiguous agree bit for bit
    assert np.array_equal(got, oracle.paged_decode(q, pool, tables, ctx, "bf16"))


def test_contiguous_rejects_out_of_range_request():
    rng = np.random.default_rng(13)
    K = W.normal_bits(rng, (2, 8, 1, 16), "bf16")
    q = W.normal_bits(rng, (1, 1, 16), "bf16")
    with pytest.raises(oracle.OracleError):
        oracle.contiguous_decode(q, K, K, np.array([2], np.int32), np.array([4], np.int32), "bf16")


def test_single_token_returns_v0_exactly():
    rng = np.random.default_rng(14)
    q, pool, tables, ctx = _tiny_paged(rng, N=2, H_q=2, H_kv=1, D=16, ctx=(1, 1))
    got = oracle.paged_decode(q, pool, tables, ctx, "bf16")
    for s in range(2):
        v0 = W.bits_to_float(pool[tables[s, 0], 0, 1, 0], "bf16").astype(np.float64)
        assert np.array_equal(got[s, 0], v0) and np.array_equal(got[s, 1], v0)


def test_zero_query_gives_mean_of_values():
    rng = np.random.default_rng(15)
    q, pool, tables, ctx = _tiny_paged(rng, N=2, H_q=2, H_kv=2, D=16, ctx=(13, 6))
    q[:] = 0
    got = oracle.paged_decode(q, pool, tables, ctx, "bf16")
    kb, vb = _gather_contiguous(pool, tables, ctx)
    for s in range(2):
        n = int(ctx[s])
        mean = W.bits_to_float(vb[s, :n], "bf16").astype(np.float64).mean(axis=0)
        np.testing.assert_allclose(got[s], mean, rtol=0, atol=1e-14)


def test_equal_value_rows_return_that_row():
    rng = np.random.default_rng(16)
    q, pool, tables, ctx = _tiny_paged(rng, N=2, H_q=2, H_kv=1, D=16, ctx=(10, 3), poison=False)
    row = W.normal_bits(rng, (16,), "bf16")
    pool[:, :, 1, 0, :] = row
    got = oracle.paged_decode(q, pool, tables, ctx, "bf16")
    np.testing.assert_allclose(got, np.broadcast_to(W.bits_to_float(row, "bf16"), got.shape), rtol=0, atol=1e-14)


def test_two_token_closed_form():
    """o = expit(x0 - x1) v0 + expit(x1 - x0) v1 with x = q.k / sqrt(D)."""
    rng = np.random.default_rng(17)
    q, pool, tables, ctx = _tiny_paged(rng, N=1, H_q=1, H_kv=1, D=16, ctx=(2,))
    got = oracle.paged_decode(q, pool, tables, ctx, "bf16")[0, 0]
    qq = W.bits_to_float(q[0, 0], "bf16").astype(np.float64)
    b = tables[0, 0]
    k0, k1 = (W.bits_to_float(pool[b, j, 0, 0], "bf16").astype(np.float64) for j in (0, 1))
    v0, v1 = (W.bits_to_float(pool[b, j, 1, 0], "bf16").astype(np.float64) for j in (0, 1))
    x0, x1 = qq @ k0 / 4.0, qq @ k1 / 4.0
    ref = scipy.special.expit(x0 - x1) * v0 + scipy.special.expit(x1 - x0) * v1
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-14)


def test_block_relabelling_leaves_output_unchanged():
    rng = np.random.default_rng(18)
    q, pool, tables, ctx = _tiny_paged(rng, N=3, H_q=4, H_kv=2, D=16, ctx=(7, 12, 30), NB=24)
    ref = oracle.paged_decode(q, pool, tables, ctx, "bf16")
    perm = rng.permutation(pool.shape[0])
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    tables2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    got = oracle.paged_decode(q, pool2, tables2, ctx, "bf16")
    assert np.array_equal(got, ref)


def test_unused_slots_are_never_read():
    rng = np.random.default_rng(19)
    q, pool, tables, ctx = _tiny_paged(rng, N=3, H_q=2, H_kv=1, D=16, ctx=(5, 6, 11), poison=True)
    got = oracle.paged_decode(q, pool, tables, ctx, "bf16")
    assert np.all(np.isfinite(got))


def test_empty_context_is_rejected():
    rng = np.random.default_rng(20)
    q, pool, tables, ctx = _tiny_paged(rng, N=1, H_q=1, H_kv=1, D=16, ctx=(3,))
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(q, pool, tables, np.array([0], np.int32), "bf16")


def test_out_of_range_table_entry_is_rejected():
    rng = np.random.default_rng(21)
    q, pool, tables, ctx = _tiny_paged(rng, N=1, H_q=1, H_kv=1, D=16, ctx=(6,))
    tables[0, 1] = pool.shape[0]
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(q, pool, tables, ctx, "bf16")


def test_pair_subset_matches_full_run():
    rng = np.random.default_rng(22)
    q, pool, tables, ctx = _tiny_paged(rng, N=3, H_q=4, H_kv=2, D=16, ctx=(4, 9, 17))
    full = oracle.paged_decode(q, pool, tables, ctx, "bf16", nthreads=2)
    pairs = np.array([[2, 3], [0, 1]], dtype=np.int32)
    sub = oracle.paged_decode(q, pool, tables, ctx, "bf16", pairs=pairs)
    for s, h in pairs:
        assert np.array_equal(sub[s, h], full[s, h])
    assert np.isnan(sub[1, 0]).all()


def test_block_streaming_pseudocode_equals_two_pass():
    rng = np.random.default_rng(23)
    q, pool, tables, ctx = _tiny_paged(rng, N=3, H_q=4, H_kv=2, D=32, B=4, NB=40, ctx=(1, 13, 31))
    ref = oracle.paged_decode(q, pool, tables, ctx, "bf16")
    for s in range(3):
        for h in range(4):
            got = oracle.paged_decode_online_row(q[s, h], pool, tables[s], ctx[s], h // 2, "bf16")
            np.testing.assert_allclose(got, ref[s, h], rtol=0, atol=1e-12)


@pytest.mark.parametrize("part", [4, 8, 12, 64])
def test_partials_merge_to_full_attention(part):
    rng = np.random.default_rng(24)
    q, pool, tables, ctx = _tiny_paged(rng, N=2, H_q=2, H_kv=1, D=16, B=4, NB=40, ctx=(29, 50))
    ref = oracle.paged_decode(q, pool, tables, ctx, "bf16")
    P = -(-int(ctx.max()) // part)
    for s in range(2):
        n = -(-int(ctx[s]) // part)
        m2, l, acc = oracle.paged_partials_row(q[s, 0], pool, tables[s], ctx[s], 0, "bf16", part, P)
        out = oracle.partition_merge(m2[None], l[None], acc[None], np.array([n], np.int32))[0]
        np.testing.assert_allclose(out, ref[s, 0], rtol=0, atol=1e-12)
        # partitions past the context are empty
        assert np.all(np.isneginf(m2[n:])) and np.all(l[n:] == 0)


def test_merge_weights_match_logsumexp():
    rng = np.random.default_rng(25)
    R, P, D = 5, 7, 8
    m2 = rng.normal(size=(R, P)) * 4
    l = rng.uniform(0.5, 3.0, size=(R, P))
    acc = rng.normal(size=(R, P, D))
    nparts = np.array([1, 3, 7, 2, 5], dtype=np.int32)
    got = oracle.partition_merge(m2, l, acc, nparts)
    for r in range(R):
        n = nparts[r]
        lnw = m2[r, :n] * np.log(2.0) + np.log(l[r, :n])
        w = np.exp(lnw - scipy.special.logsumexp(lnw))        # share of each partition in the normaliser
        ref = (w[:, None] * acc[r, :n] / l[r, :n, None]).sum(axis=0)
        np.testing.assert_allclose(got[r], ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- cache ops

def test_reshape_and_cache_matches_numpy_indexing():
    rng = np.random.default_rng(30)
    NB, B, H, D, T = 12, 4, 3, 16, 20
    pool = W.normal_bits(rng, (NB, B, 2, H, D), "f16")
    ref = pool.copy()
    k = W.normal_bits(rng, (T, H, D), "f16")
    v = W.normal_bits(rng, (T, H, D), "f16")
    slots = rng.choice(NB * B, size=T, replace=False).astype(np.int64)
    slots[[3, 11]] = -1
    oracle.reshape_and_cache(k, v, pool, slots)
    keep = slots >= 0
    ref[slots[keep] // B, slots[keep] % B, 0] = k[keep]
    ref[slots[keep] // B, slots[keep] % B, 1] = v[keep]
    assert np.array_equal(pool, ref)


def test_reshape_and_cache_rejects_out_of_range_slot():
    rng = np.random.default_rng(31)
    pool = W.normal_bits(rng, (2, 4, 2, 1, 16), "f16")
    k = W.normal_bits(rng, (1, 1, 16), "f16")
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(k, k, pool, np.array([8], np.int64))


def test_copy_blocks_matches_numpy_copy():
    rng = np.random.default_rng(32)
    pool = W.normal_bits(rng, (10, 4, 2, 2, 16), "bf16")
    ref = pool.copy()
    pairs = np.array([[1, 7], [3, 0], [1, 9]], dtype=np.int64)
    oracle.copy_blocks(pool, pairs)
    for s, d in pairs:
        ref[d] = ref[s]
    assert np.array_equal(pool, ref)


@pytest.mark.parametrize("pairs", [[[1, 2], [2, 3]], [[1, 2], [4, 2]], [[5, 5]], [[0, 10]]])
def test_copy_blocks_rejects_chained_duplicate_or_out_of_range(pairs):
    rng = np.random.default_rng(33)
    pool = W.normal_bits(rng, (10, 4, 2, 1, 16), "bf16")
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(pool, np.array(pairs, dtype=np.int64))


def test_rows_listed_twice_are_computed_correctly_in_parallel():
    rng = np.random.default_rng(26)
    q, pool, tables, ctx = _tiny_paged(rng, N=2, H_q=2, H_kv=1, D=16, ctx=(37, 29))
    full = oracle.paged_decode(q, pool, tables, ctx, "bf16")
    pairs = np.array([[0, 1]] * 16 + [[1, 0]] * 16, dtype=np.int32)
    for _ in range(5):
        sub = oracle.paged_decode(q, pool, tables, ctx, "bf16", pairs=pairs, nthreads=8)
        assert np.array_equal(sub[0, 1], full[0, 1]) and np.array_equal(sub[1, 0], full[1, 0])


def test_swap_blocks_matches_numpy_copy_between_pools():
    rng = np.random.default_rng(34)
    dev = W.normal_bits(rng, (12, 4, 2, 2, 16), "bf16")
    host = W.normal_bits(rng, (7, 4, 2, 2, 16), "bf16")
    ref = host.copy()
    pairs = np.array([[3, 6], [11, 0], [3, 2]], dtype=np.int64)
    oracle.swap_blocks(host, dev, pairs)
    for s, d in pairs:
        ref[d] = dev[s]
    assert np.array_equal(host, ref)
    for bad in ([[0, 7]], [[12, 0]], [[1, 2], [3, 2]]):
        with pytest.raises(oracle.OracleError):
            oracle.swap_blocks(host, dev, np.array(bad, dtype=np.int64))


# ----------------------------------------------------------------------------- prefill

def _prefill_case(rng, chunks, ctx, H_q=4, H_kv=2, D=16, B=4, NB=80, dtype="bf16"):
    q_dummy, pool, tables, ctx = _tiny_paged(rng, N=len(ctx), H_q=H_q, H_kv=H_kv, D=D, B=B, NB=NB, dtype=dtype,
                                             ctx=ctx)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = W.normal_bits(rng, (int(q_start[-1]), H_q, D), dtype)
    return q, pool, tables, ctx, q_start


def test_prefill_matches_library_causal_attention():
    """Full prefill (chunk = whole sequence) equals torch SDPA with a causal mask in fp64; a chunk equals the
    last rows of the full causal attention."""
    rng = np.random.default_rng(40)
    ctx = (9, 17, 6)
    chunks = (9, 5, 1)
    q, pool, tables, ctx, q_start = _prefill_case(rng, chunks, ctx)
    got = oracle.paged_prefill(q, pool, tables, ctx, q_start, "bf16", nthreads=2)
    kb, vb = _gather_contiguous(pool, tables, ctx)
    for s, n in enumerate(ctx):
        ql = int(q_start[s + 1] - q_start[s])
        G = 2
        k = torch.from_numpy(W.bits_to_float(kb[s, :n], "bf16").astype(np.float64)).permute(1, 0, 2)
        v = torch.from_numpy(W.bits_to_float(vb[s, :n], "bf16").astype(np.float64)).permute(1, 0, 2)
        k, v = k.repeat_interleave(G, 0), v.repeat_interleave(G, 0)
        qq = torch.from_numpy(W.bits_to_float(q[q_start[s]:q_start[s + 1]], "bf16").astype(np.float64))
        # queries sit at the last ql positions: build the [H, ql, n] causal mask explicitly
        pos = np.arange(n - ql, n)[:, None]
        mask = torch.from_numpy(np.arange(n)[None, :] <= pos)
        ref = torch.nn.functional.scaled_dot_product_attention(qq.permute(1, 0, 2), k, v, attn_mask=mask)
        np.testing.assert_allclose(got[q_start[s]:q_start[s + 1]], ref.permute(1, 0, 2).numpy(), rtol=0,
                                   atol=1e-12)


def test_prefill_of_one_token_is_decode():
    rng = np.random.default_rng(41)
    q, pool, tables, ctx, q_start = _prefill_case(rng, (1, 1, 1), (7, 13, 4))
    pre = oracle.paged_prefill(q, pool, tables, ctx, q_start, "bf16")
    dec = oracle.paged_decode(q, pool, tables, ctx, "bf16")
    assert np.array_equal(pre, dec)


def test_prefill_first_position_returns_its_own_value():
    rng = np.random.default_rng(42)
    q, pool, tables, ctx, q_start = _prefill_case(rng, (5,), (5,), H_q=2, H_kv=1)
    got = oracle.paged_prefill(q, pool, tables, ctx, q_start, "bf16")
    v0 = W.bits_to_float(pool[tables[0, 0], 0, 1, 0], "bf16").astype(np.float64)
    assert np.array_equal(got[0, 0], v0) and np.array_equal(got[0, 1], v0)
