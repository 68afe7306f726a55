"""Pins for the oracle's block-allocator model (no GPU).

The worked block-table example and the fragmentation bound come from the
PagedAttention explainer; the copy-on-write count of the parallel-sampling
workload follows from the copy-before-write rule applied in sample order.
"""
import os

import numpy as np
import pytest

import workloads as W
from oracle.alloc_model import AllocError, AllocModel

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_worked_example():
    tables, slots, tokens, B = {}, {}, {}, None
    with open(os.path.join(GOLDEN, "worked_example.txt")) as f:
        for line in f:
            p = line.split()
            if not p or p[0].startswith("#"):
                continue
            if p[0] == "block_size":
                B = int(p[1])
            elif p[0] == "table":
                tables[p[1]] = [int(x) for x in p[2:]]
            elif p[0] == "slots":
                slots[p[1]] = [int(x) for x in p[2:]]
            elif p[0] == "tokens":
                tokens[p[1]] = int(p[2])
    return B, tables, slots, tokens


def test_worked_example_tables_and_slots():
    B, tables, slots, tokens = _read_worked_example()
    w = W.tiny()
    assert w.B == B
    m = AllocModel(w.NB, w.B, w.free_order)
    got_slots = {}
    for s, name in enumerate(["A", "B", "C", "D"]):
        m.add_seq(s)
        got_slots[name], cow = m.append_slots(s, int(w.ctx[s]))
        assert cow == []
    assert int(w.ctx[0]) == tokens["A"] and int(w.ctx[1]) == tokens["B"]
    assert m.block_table(0) == tables["A"] and m.block_table(1) == tables["B"]
    assert got_slots["A"] == slots["A"] and got_slots["B"] == slots["B"]


def _invariants(m: AllocModel):
    used = set()
    refsum = 0
    for seq, tab in m.tables.items():
        n = m.ntok[seq]
        assert len(tab) == -(-n // m.B)
        # internal fragmentation of a request is at most B-1 tokens
        assert len(tab) * m.B - n <= m.B - 1
        refsum += len(tab)
        used.update(tab)
    assert refsum == sum(m.ref)
    assert len(m.free) + len(used) == m.NB
    assert not (set(m.free) & used)
    assert all(m.ref[b] == 0 for b in m.free)


def test_random_operation_sequences_keep_invariants():
    rng = np.random.default_rng(40)
    for trial in range(20):
        NB, B = int(rng.integers(8, 80)), int(rng.choice([1, 2, 4, 8, 16]))
        m = AllocModel(NB, B, rng.permutation(NB))
        live, nxt = [], 0
        for _ in range(300):
            op = rng.integers(0, 4)
            try:
                if op == 0 or not live:
                    m.add_seq(nxt)
                    live.append(nxt)
                    nxt += 1
                elif op == 1:
                    s = live[rng.integers(len(live))]
                    before = (list(m.free), list(m.ref), {k: list(v) for k, v in m.tables.items()})
                    try:
                        slots, cow = m.append_slots(s, int(rng.integers(0, 3 * B + 2)))
                    except AllocError as e:
                        assert e.kind == "oom"
                        assert before == (m.free, m.ref, m.tables)   # all-or-nothing
                        continue
                    for old, new in cow:
                        assert m.ref[new] == 1 and new in m.tables[s]
                elif op == 2:
                    s = live[rng.integers(len(live))]
                    m.fork(s, nxt)
                    live.append(nxt)
                    nxt += 1
                else:
                    s = live.pop(rng.integers(len(live)))
                    m.free_seq(s)
            finally:
                _invariants(m)


def test_cow_workload_emits_one_copy_per_sample_but_the_last():
    w = W.cow(prompts=4, samples=8)
    m = AllocModel(w.NB, w.B, w.free_order)
    pairs = []
    for p in range(w.prompts):
        base = p * w.samples
        m.add_seq(base)
        m.append_slots(base, w.prompt_len)
        for j in range(1, w.samples):
            m.fork(base, base + j)
        last = m.block_table(base)[-1]
        assert m.refcount(last) == w.samples
    for s in range(w.N):
        slots, cow = m.append_slots(s, int(w.extra[s]))
        pairs += cow
        # after the write every block the sample writes into is private
        for slot in slots:
            assert m.refcount(slot // w.B) == 1
    # 1030 = 64*16 + 6: the shared last block is partial, so samples 0..6 copy and sample 7 writes in place
    assert w.prompt_len % w.B != 0
    assert len(pairs) == w.prompts * (w.samples - 1)
    _invariants(m)


def test_full_cow_workload_has_224_pairs():
    w = W.cow()
    m = AllocModel(w.NB, w.B, w.free_order)
    n = 0
    for p in range(w.prompts):
        base = p * w.samples
        m.add_seq(base)
        m.append_slots(base, w.prompt_len)
        for j in range(1, w.samples):
            m.fork(base, base + j)
    for s in range(w.N):
        n += len(m.append_slots(s, int(w.extra[s]))[1])
    assert n == 224


def test_free_pushes_blocks_in_logical_order():
    m = AllocModel(6, 2, [0, 1, 2, 3, 4, 5])
    m.add_seq(0)
    m.append_slots(0, 5)          # blocks 0, 1, 2
    assert m.block_table(0) == [0, 1, 2]
    m.free_seq(0)
    assert m.free_list_top_first()[:3] == [2, 1, 0]


def test_errors():
    m = AllocModel(2, 4)
    with pytest.raises(AllocError):
        m.append_slots(0, 1)
    m.add_seq(0)
    with pytest.raises(AllocError):
        m.add_seq(0)
    with pytest.raises(AllocError) as e:
        m.append_slots(0, 9)
    assert e.value.kind == "oom" and m.seq_len(0) == 0 and m.num_free() == 2
    with pytest.raises(AllocError):
        m.fork(1, 2)
    with pytest.raises(AllocError):
        AllocModel(3, 4, [0, 0, 1])


def _apply(m, op):
    kind = op[0]
    if kind == "add":
        m.add_seq(op[1])
    elif kind == "append":
        return m.append_slots(op[1], op[2])
    elif kind == "fork":
        m.fork(op[1], op[2])
    elif kind == "free":
        m.free_seq(op[1])
    return None


def test_beam_search_fork_tree_shares_prefixes_and_copies_on_write():
    """Beams forked from beams share every common prefix block; each shared block's count equals the
    number of live beams whose table holds it, and a write never lands in a block another beam reads."""
    ops = W.beam_search_ops()
    m = AllocModel(256, 16, np.random.default_rng(7).permutation(256))
    copies = 0
    for op in ops:
        if op[0] == "round_end":
            live = op[1]
            holders = {}
            for b in live:
                for blk in m.block_table(b):
                    holders[blk] = holders.get(blk, 0) + 1
            assert all(m.refcount(blk) == n for blk, n in holders.items())
            assert len(m.tables) == len(live)
            # the prompt's first full block is shared by every live beam
            assert holders[m.block_table(live[0])[0]] == len(live)
            _invariants(m)
            continue
        res = _apply(m, op)
        if res is not None:
            slots, cow = res
            copies += len(cow)
            for s in slots:
                assert m.refcount(s // m.B) == 1
    assert copies > 0
