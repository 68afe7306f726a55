"""Host-side checks of libpa.so (no GPU): symbol exports, argument validation,
and the C++ block allocator against the oracle's independent model."""
import ctypes

import numpy as np
import pytest

import paged_kv_cache_302_gb300 as pa
import workloads as W
from oracle.alloc_model import AllocError, AllocModel


def test_library_exports_every_declared_function():
    L = pa.load()
    names = pa.header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), n
    assert "sm_103a" in pa.version()


def test_workspace_sizes():
    assert pa.pa_decode_workspace_bytes(256, 32, 8, 128, 8192, 0) > 256 * 32 * 16 * 128 * 4
    small = pa.pa_decode_workspace_bytes(4, 2, 2, 64, 33, -1)
    assert 0 < small < 4096
    for bad in [(0, 1, 1, 128, 10, 0), (1, 1, 1, 128, 10, 48), (1, 1, 1, 128, 0, 0)]:
        with pytest.raises(pa.PAError):
            pa.pa_decode_workspace_bytes(*bad)


def test_device_calls_reject_bad_arguments_before_touching_the_gpu():
    L = pa.load()
    # unsupported dtype / bad sizes are refused by host validation
    assert L.pa_reshape_and_cache(None, None, None, None, 1, 4, 4, 1, 8, 2, None, None) == pa.PA_ERR_UNSUPPORTED
    assert L.pa_reshape_and_cache(None, None, None, None, -1, 4, 4, 1, 8, 1, None, None) == pa.PA_ERR_INVALID
    assert L.pa_reshape_and_cache(None, None, None, None, 0, 4, 4, 1, 8, 1, None, None) == pa.PA_OK
    assert L.pa_copy_blocks(None, None, 0, 4, 4, 1, 8, 1, None, None) == pa.PA_OK
    assert L.pa_copy_blocks(None, None, 3, 4, 4, 1, 8, 1, None, None) == pa.PA_ERR_INVALID
    st = L.pa_decode(None, 2, None, None, None, None, 1, 16, 1, 128, 16, 1, 1, 16, 0.1, 0, None, 0, 1, None, None,
                     None)
    assert st == pa.PA_ERR_UNSUPPORTED and "H_q / H_kv" in pa.last_error()
    st = L.pa_decode(None, 2, None, None, None, None, 1, 2, 1, 96, 16, 1, 1, 16, 0.1, 0, None, 0, 1, None, None,
                     None)
    assert st == pa.PA_ERR_UNSUPPORTED
    st = L.pa_decode(None, 0, None, None, None, None, 1, 2, 1, 128, 16, 1, 1, 16, 0.1, 0, None, 0, 1, None, None,
                     None)
    assert st == pa.PA_ERR_UNSUPPORTED and "out_dtype" in pa.last_error()
    st = L.pa_partition_reduce(None, 2, None, None, None, None, 0, 4, 128, None, None)
    assert st == pa.PA_OK
    # pa_prefill: placeholder addresses are never dereferenced because validation fails first
    out, q, pool, tab, ctx, qs = 0x1010, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000

    def prefill(out=out, out_dtype=2, B=16, scale=0.1, ws=None):
        return L.pa_prefill(out, out_dtype, q, pool, tab, ctx, qs, 1, 1, 8, 8, 128, B, 1, 1, 1, scale, 1, ws, 0,
                            None, None)

    assert prefill() == pa.PA_ERR_INVALID and "32-byte" in pa.last_error()
    assert prefill(out=0x1008, out_dtype=1) == pa.PA_ERR_INVALID and "16-byte" in pa.last_error()
    assert prefill(out=0x1020, ws=0x7008) == pa.PA_ERR_INVALID and "16-byte" in pa.last_error()
    assert prefill(out=0x1020, B=4) == pa.PA_ERR_UNSUPPORTED
    assert prefill(out=0x1020, scale=0.0) == pa.PA_ERR_INVALID
    # the prefill workspace: staged V [N * H_kv][S_pad][D] 16-bit (S_pad = MB * B rounded up to 128 keys), then
    # one flag byte per 32 keys, each part rounded up to 256 bytes
    assert L.pa_prefill_workspace_bytes(2, 8, 128, 16, 10) == 2 * 8 * 256 * 128 * 2 + 256
    assert L.pa_prefill_workspace_bytes(3, 1, 64, 8, 17) == 3 * 256 * 64 * 2 + 256
    assert L.pa_prefill_workspace_bytes(0, 8, 128, 16, 10) == 0 and L.pa_prefill_workspace_bytes(1, 8, 96, 16, 1) == 0


def _run_same_ops(NB, B, order, ops):
    """Apply the same operation list to the C++ allocator and the model; compare every observable."""
    cpp = pa.BlockAllocator(NB, B, order)
    ref = AllocModel(NB, B, order)
    live = set()
    for op in ops:
        kind = op[0]
        got_err = want_err = None
        try:
            if kind == "add":
                cpp.add_seq(op[1])
        except pa.PAError as e:
            got_err = e.status
        try:
            if kind == "add":
                ref.add_seq(op[1])
        except AllocError as e:
            want_err = e.kind
        if kind == "append":
            try:
                got = cpp.append_slots(op[1], op[2])
            except pa.PAError as e:
                got_err, got = e.status, None
            try:
                want = ref.append_slots(op[1], op[2])
            except AllocError as e:
                want_err, want = e.kind, None
            if got is not None and want is not None:
                assert list(got[0]) == want[0]
                assert [tuple(r) for r in got[1]] == want[1]
        elif kind == "batch":
            try:
                got = cpp.append_batch(op[1], op[2], table_updates=True)
            except pa.PAError as e:
                got_err, got = e.status, None
            snapshot = (list(ref.free), list(ref.ref), {k: list(v) for k, v in ref.tables.items()}, dict(ref.ntok))
            try:
                slots, pairs, upd = [], [], []
                for row, (s, n) in enumerate(zip(op[1], op[2])):
                    before = list(ref.tables[s]) if s in ref.tables else []
                    a, b = ref.append_slots(s, n)
                    slots += a
                    pairs += b
                    after = ref.tables[s]
                    # table entries that changed or appeared, in logical order
                    upd += [(row, lb, after[lb]) for lb in range(len(after))
                            if lb >= len(before) or before[lb] != after[lb]]
                want = (slots, pairs, upd)
            except AllocError as e:
                want_err, want = e.kind, None
                ref.free, ref.ref, ref.tables, ref.ntok = snapshot      # the batch is all-or-nothing
            if got is not None and want is not None:
                assert list(got[0]) == want[0]
                assert [tuple(r) for r in got[1]] == want[1]
                assert [tuple(int(x) for x in r) for r in got[2]] == want[2]
        elif kind == "fork":
            try:
                cpp.fork(op[1], op[2])
            except pa.PAError as e:
                got_err = e.status
            try:
                ref.fork(op[1], op[2])
            except AllocError as e:
                want_err = e.kind
        elif kind == "free":
            try:
                cpp.free_seq(op[1])
            except pa.PAError as e:
                got_err = e.status
            try:
                ref.free_seq(op[1])
            except AllocError as e:
                want_err = e.kind
        kinds = {None: None, "invalid": pa.PA_ERR_INVALID, "oom": pa.PA_ERR_OOM, "state": pa.PA_ERR_STATE}
        assert got_err == kinds[want_err], (op, got_err, want_err)
        # full state comparison
        assert cpp.num_free() == ref.num_free()
        assert list(cpp.free_list()) == ref.free_list_top_first()
        for s in ref.tables:
            assert list(cpp.block_table(s)) == ref.block_table(s)
            assert cpp.seq_len(s) == ref.seq_len(s)
        for b in range(NB):
            assert cpp.refcount(b) == ref.refcount(b)
    cpp.close()


def test_allocator_matches_model_on_worked_example():
    w = W.tiny()
    ops = [("add", s) for s in range(4)] + [("append", s, int(w.ctx[s])) for s in range(4)]
    _run_same_ops(w.NB, w.B, w.free_order, ops)
    a = pa.BlockAllocator(w.NB, w.B, w.free_order)
    for s in range(4):
        a.add_seq(s)
        a.append_slots(s, int(w.ctx[s]))
    assert list(a.block_table(0)) == [7, 1] and list(a.block_table(1)) == [3, 5]


def test_allocator_matches_model_on_random_operations():
    rng = np.random.default_rng(50)
    for trial in range(12):
        NB = int(rng.integers(6, 60))
        B = int(rng.choice([1, 2, 4, 8, 16]))
        ops, nxt, live = [], 0, []
        for _ in range(150):
            r = rng.integers(0, 10)
            if r < 2 or not live:
                ops.append(("add", nxt))
                live.append(nxt)
                nxt += 1
            elif r < 5:
                ops.append(("append", int(rng.choice(live + [999])), int(rng.integers(-1, 3 * B + 2))))
            elif r < 7:
                k = int(rng.integers(1, len(live) + 1))
                ids = [int(x) for x in rng.choice(live, size=k, replace=False)]
                ops.append(("batch", ids, [int(x) for x in rng.integers(0, 2 * B + 2, size=k)]))
            elif r < 8:
                ops.append(("fork", int(rng.choice(live)), nxt))
                live.append(nxt)
                nxt += 1
            else:
                s = int(rng.choice(live))
                live.remove(s)
                ops.append(("free", s))
        ops = [o for o in ops if not (o[0] == "append" and o[2] < 0)]
        _run_same_ops(NB, B, rng.permutation(NB), ops)


def test_allocator_cow_workload_matches_model():
    w = W.cow(prompts=3, samples=8, prompt_len=1030)
    ops = []
    for p in range(w.prompts):
        base = p * w.samples
        ops += [("add", base), ("append", base, w.prompt_len)]
        ops += [("fork", base, base + j) for j in range(1, w.samples)]
    ops.append(("batch", list(range(w.N)), [int(x) for x in w.extra]))
    _run_same_ops(w.NB, w.B, w.free_order, ops)


def test_allocator_errors():
    a = pa.BlockAllocator(2, 4)
    with pytest.raises(pa.PAError) as e:
        a.append_slots(0, 1)
    assert e.value.status == pa.PA_ERR_INVALID
    a.add_seq(0)
    with pytest.raises(pa.PAError) as e:
        a.append_slots(0, 9)
    assert e.value.status == pa.PA_ERR_OOM and a.num_free() == 2 and a.seq_len(0) == 0
    with pytest.raises(pa.PAError):
        a.append_batch([0, 0], [1, 1])
    with pytest.raises(pa.PAError):
        pa.BlockAllocator(3, 4, [0, 0, 1])
    L = pa.load()
    assert L.pa_alloc_num_free(None) == -1
    h = ctypes.c_void_p()
    assert L.pa_alloc_create(0, 4, None, ctypes.byref(h)) == pa.PA_ERR_INVALID


def test_block_tables_packing():
    a = pa.BlockAllocator(16, 4, list(range(16)))
    for s, n in [(0, 5), (1, 9), (2, 1)]:
        a.add_seq(s)
        a.append_slots(s, n)
    tab, ctx = a.block_tables([2, 0, 1], 4)
    assert list(ctx) == [1, 5, 9]
    assert list(tab[0]) == [5, -1, -1, -1]
    assert list(tab[1]) == [0, 1, -1, -1]
    assert list(tab[2]) == [2, 3, 4, -1]
    with pytest.raises(pa.PAError):
        a.block_tables([1], 2)


def test_allocator_matches_model_on_beam_search_fork_tree():
    ops = [o for o in W.beam_search_ops() if o[0] != "round_end"]
    _run_same_ops(256, 16, np.random.default_rng(7).permutation(256), ops)


def test_swap_rejects_pageable_host_memory_before_any_launch():
    L = pa.load()
    host = np.zeros((4, 16, 2, 1, 64), dtype=np.uint16)
    pairs = np.zeros((1, 2), dtype=np.int64)
    st = L.pa_swap_blocks(host.ctypes.data, 4, host.ctypes.data, 4, pairs.ctypes.data, 1, 16, 1, 64, 1, None, None)
    assert st in (pa.PA_ERR_INVALID, pa.PA_ERR_CUDA)


def test_nvtx_ranges_can_be_switched_on():
    """PA_NVTX=1 wraps every device call in an NVTX range (a no-op without a profiler attached)."""
    import os
    import subprocess
    import sys
    code = ("import paged_kv_cache_302_gb300 as pa; L = pa.load(); "
            "st = L.pa_decode(None, 2, None, None, None, None, 1, 16, 1, 128, 16, 1, 1, 16, 0.1, 0, None, 0, 1, "
            "None, None, None); assert st == pa.PA_ERR_UNSUPPORTED, st; "
            "assert L.pa_reshape_and_cache(None, None, None, None, 0, 4, 4, 1, 8, 1, None, None) == pa.PA_OK")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=dict(os.environ, PA_NVTX="1"),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr


def _observe(a, ids):
    return (list(a.free_list()), a.num_free(), [list(a.block_table(s)) for s in ids], [a.seq_len(s) for s in ids],
            [a.refcount(b) for b in range(a.NB)])


def _mixed_state(NB=48, B=4, seed=60):
    rng = np.random.default_rng(seed)
    a = pa.BlockAllocator(NB, B, rng.permutation(NB))
    for s in range(4):
        a.add_seq(s)
        a.append_slots(s, int(rng.integers(1, 11)))
    a.fork(0, 10)
    a.fork(10, 11)                      # a shared partial block with count 3
    a.append_slots(11, 3)               # copy-on-write
    a.free_seq(2)
    return a, [0, 1, 3, 10, 11]


def test_allocator_state_round_trips_and_continues_identically():
    a, ids = _mixed_state()
    state = a.export_state()
    b = pa.BlockAllocator.from_state(state)
    assert _observe(b, ids) == _observe(a, ids)
    assert np.array_equal(b.export_state(), state)
    for x in (a, b):                    # the same operations on the original and the resumed allocator
        x.append_slots(0, 5)
        x.add_seq(20)
        x.append_slots(20, 9)
        x.fork(20, 21)
        x.free_seq(1)
    for s in (0, 20, 21, 10, 11):
        assert list(a.append_slots(s, 2)[0]) == list(b.append_slots(s, 2)[0])
    ids = [0, 3, 10, 11, 20, 21]
    assert _observe(b, ids) == _observe(a, ids)


def test_allocator_import_rejects_inconsistent_states():
    a, _ = _mixed_state()
    good = a.export_state()
    NB, nfree = int(good[1]), int(good[3])
    free0, ref0 = 5, 5 + nfree
    used = [b for b in range(NB) if good[ref0 + b] > 0]

    def bad(mut):
        s = good.copy()
        s = mut(s)
        with pytest.raises(pa.PAError) as e:
            pa.BlockAllocator.from_state(s)
        assert e.value.status == pa.PA_ERR_INVALID

    bad(lambda s: np.concatenate([[0], s[1:]]))                            # not a state
    bad(lambda s: np.concatenate([s, [0]]))                                # trailing word
    bad(lambda s: s[:-1])                                                  # truncated
    def dup_free(s):
        s[free0 + 1] = s[free0]
        return s
    bad(dup_free)                                                          # a block listed free twice
    def ref_off(s):
        s[ref0 + used[0]] += 1
        return s
    bad(ref_off)                                                           # count disagrees with the tables
    def drop_free(s):
        s[3] -= 1
        return np.delete(s, free0)
    bad(drop_free)                                                         # a block neither free nor used
    def wrong_len(s):
        seq0 = ref0 + NB
        s[seq0 + 1] += 4 * int(s[2])                                       # tokens no longer match the blocks
        return s
    bad(wrong_len)
