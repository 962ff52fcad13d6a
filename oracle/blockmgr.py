"""Oracle block manager: a plain restatement of the paged pool's bookkeeping.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows, in this order:
  * "llm-inference-batching" (faangrind), the KV pool listing: a free list of
    block ids, a block table per request, and ref_count[block] that is above
    1 when samples or a prompt share the block;
  * "continuous batching server" (scalablesystem), "The KV Cache Block
    Manager": blocks_needed = ceil(tokens / 16), blocks taken with a pop from
    the end of the free list and returned by extending it;
  * "Serving LLMs" (sreshtalluri), "Paged KV memory": growing a request that
    needs more blocks than are free fails with no change, which is the
    signal to preempt;
  * "The inference engine" (wpnews), "Paging turns variable sequences into
    block tables": sequences may point at the same immutable prefix blocks.

Status codes use the library's numbering so the two can be compared directly.
"""
from __future__ import annotations

OK, E_INVALID, E_NOMEM, E_SHARED = 0, 1, 2, 3


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int = 16, free_order=None):
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        assert sorted(order) == list(range(num_blocks))
        self.block_size = block_size
        self.num_blocks = num_blocks
        self.free = list(reversed(order))        # the end of the list is handed out next
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}

    def blocks_needed(self, tokens: int) -> int:
        return -(-tokens // self.block_size)

    def grow(self, seq: int, new_len: int) -> int:
        table = self.tables.get(seq, [])
        if new_len < self.lens.get(seq, 0) or new_len < 0:
            return E_INVALID
        need = self.blocks_needed(new_len) - len(table)
        if need > len(self.free):
            return E_NOMEM
        for _ in range(max(need, 0)):
            b = self.free.pop()
            self.ref[b] = 1
            table.append(b)
        self.tables[seq] = table
        self.lens[seq] = new_len
        return OK

    def share_prefix(self, dst: int, src: int, n_blocks: int) -> int:
        if src not in self.tables or dst in self.tables or dst == src:
            return E_INVALID
        if n_blocks < 0 or n_blocks * self.block_size > self.lens[src]:
            return E_INVALID
        shared = self.tables[src][:n_blocks]
        for b in shared:
            self.ref[b] += 1
        self.tables[dst] = list(shared)
        self.lens[dst] = n_blocks * self.block_size
        return OK

    def free_seq(self, seq: int) -> int:
        if seq not in self.tables:
            return E_INVALID
        for b in self.tables.pop(seq):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        del self.lens[seq]
        return OK

    def free_blocks(self) -> int:
        return len(self.free)

    def build_step(self, seqs, q_lens, max_blocks: int):
        """Step metadata: (status, tables, ctx_lens, slots, q_start_loc).

        Row i's new tokens are its last q_lens[i] positions; each must land in
        a block this sequence owns alone (ref_count 1)."""
        tables = [[-1] * max_blocks for _ in seqs]
        ctx, slots, qstart = [], [], [0]
        for i, (s, q) in enumerate(zip(seqs, q_lens)):
            if s not in self.tables or q < 1 or q > self.lens[s]:
                return E_INVALID, None, None, None, None
            t = self.tables[s]
            if len(t) > max_blocks:
                return E_INVALID, None, None, None, None
            n = self.lens[s]
            tables[i][:len(t)] = t
            ctx.append(n)
            for p in range(n - q, n):
                b = t[p // self.block_size]
                if self.ref[b] != 1:
                    return E_SHARED, None, None, None, None
                slots.append(b * self.block_size + p % self.block_size)
            qstart.append(qstart[-1] + q)
        return OK, tables, ctx, slots, qstart
