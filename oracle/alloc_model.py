"""Independent model of the paged-KV block allocator (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources (page titles and sections):
  "論文解説: PagedAttention — 仮想メモリ着想のKVキャッシュ管理でLLMサービングを高効率化"
  * 技術的詳細 / PagedAttentionアルゴリズム: a sequence of T tokens uses ceil(T/B)
    fixed-size blocks that can sit anywhere; a per-sequence block table maps
    logical block -> physical block (the worked example: Request A, 7 tokens,
    B=4 -> blocks 7, 1; Request B, 5 tokens -> 3, 5).
  * 技術的詳細 / Copy-on-Write KVキャッシュ共有: a shared block carries a reference
    count equal to the number of sequences using it; a write into a block whose
    count exceeds one copies the block first.
  * 実装のポイント: blocks come from one slab with the library's own allocator,
    allocated on demand and freed when a request finishes.

Readings where the pages are silent (each is listed in the design notes):
  * free list: a LIFO stack.  ``initial_free_order`` lists block ids in the
    order they are handed out (first entry first).  Freeing pushes a
    sequence's blocks in logical order, so its last block is reused first.
  * slot of token position ``pos``: physical_block(pos // B) * B + pos % B.
  * copy-on-write: when a token lands in a non-empty last block whose count is
    above one, a fresh block is taken, the pair (old, new) is emitted for the
    device copy, the old count drops by one and the table points at the new
    block.  A token that starts a new block never copies.
  * every operation is all-or-nothing: running out of blocks leaves the state
    unchanged.
"""
from __future__ import annotations


class AllocError(RuntimeError):
    def __init__(self, kind: str, msg: str):
        super().__init__(f"{kind}: {msg}")
        self.kind = kind


class AllocModel:
    def __init__(self, num_blocks: int, block_size: int, initial_free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise AllocError("invalid", "sizes must be positive")
        order = list(range(num_blocks)) if initial_free_order is None else [int(b) for b in initial_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise AllocError("invalid", "initial_free_order must be a permutation of 0..NB-1")
        self.NB = num_blocks
        self.B = block_size
        self.free = order[::-1]          # stack; the top is the end of the list
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.ntok: dict[int, int] = {}

    # ------------------------------------------------------------------ queries
    def num_free(self) -> int:
        return len(self.free)

    def free_list_top_first(self) -> list[int]:
        return self.free[::-1]

    def block_table(self, seq: int) -> list[int]:
        self._need(seq)
        return list(self.tables[seq])

    def seq_len(self, seq: int) -> int:
        self._need(seq)
        return self.ntok[seq]

    def refcount(self, block: int) -> int:
        if not 0 <= block < self.NB:
            raise AllocError("invalid", "block out of range")
        return self.ref[block]

    # ------------------------------------------------------------------ operations
    def add_seq(self, seq: int):
        if seq < 0 or seq in self.tables:
            raise AllocError("invalid", f"sequence {seq} exists or is negative")
        self.tables[seq] = []
        self.ntok[seq] = 0

    def append_slots(self, seq: int, n: int):
        """Append n tokens; returns (slots, cow_pairs)."""
        self._need(seq)
        if n < 0:
            raise AllocError("invalid", "negative token count")
        table, pos = self.tables[seq], self.ntok[seq]
        # how many fresh blocks this call needs (new blocks plus at most one copy)
        need = 0
        if n > 0 and pos % self.B != 0 and self.ref[table[-1]] > 1:
            need += 1
        first_new = -(-pos // self.B)            # ceil(pos / B): blocks already covering [0, pos)
        last_needed = -(-(pos + n) // self.B)
        need += max(0, last_needed - first_new)
        if need > len(self.free):
            raise AllocError("oom", f"need {need} blocks, {len(self.free)} free")
        slots, cow = [], []
        for _ in range(n):
            off = pos % self.B
            if off == 0:
                b = self.free.pop()
                self.ref[b] = 1
                table.append(b)
            elif self.ref[table[-1]] > 1:
                old = table[-1]
                b = self.free.pop()
                self.ref[b] = 1
                self.ref[old] -= 1
                table[-1] = b
                cow.append((old, b))
            slots.append(table[pos // self.B] * self.B + off)
            pos += 1
        self.ntok[seq] = pos
        return slots, cow

    def fork(self, parent: int, child: int):
        self._need(parent)
        if child < 0 or child in self.tables:
            raise AllocError("invalid", f"child {child} exists or is negative")
        self.tables[child] = list(self.tables[parent])
        self.ntok[child] = self.ntok[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_seq(self, seq: int):
        self._need(seq)
        for b in self.tables[seq]:
            if self.ref[b] <= 0:
                raise AllocError("state", f"block {b} has no reference")
        for b in self.tables[seq]:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        del self.tables[seq]
        del self.ntok[seq]

    def _need(self, seq: int):
        if seq not in self.tables:
            raise AllocError("invalid", f"unknown sequence {seq}")
