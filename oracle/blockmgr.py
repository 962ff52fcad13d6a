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
    block tables": sequences may point at the same immutable prefix blocks,
    and copy-on-write restores separate ownership when a branch diverges
    (fork shares every block; before a step writes positions that fall in
    a block another sequence also holds, cow gives the writer a private copy
    of that block);
  * "continuous batching server", "Preemption and Eviction: Recompute vs
    Swap": a swapped-out victim keeps its length but gives its blocks back;
    swapping in allocates fresh blocks for the host copy to return to;
  * "Serving LLMs" (sreshtalluri), "Prefix caching": full blocks are keyed by
    a chained hash (the oracle's block_hashes); a lookup walks the chain
    until the first miss; the cache holds one reference per cached block.
    Reading for eviction (the page names LRU for a radix-tree variant): an
    entry whose block only the cache still references may be evicted, least
    recently used first, deeper chain positions first among equals.

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
        self.swapped: set[int] = set()
        self.cache: dict[int, list] = {}          # hash -> [block, last_use, depth]
        self.cached_blocks: set[int] = set()      # a block is cached under one hash at most
        self.clock = 0

    def blocks_needed(self, tokens: int) -> int:
        return -(-tokens // self.block_size)

    def grow(self, seq: int, new_len: int) -> int:
        if seq in self.swapped:
            return E_INVALID
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
        if src not in self.tables or dst in self.tables or dst == src or src in self.swapped:
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
        self.swapped.discard(seq)
        return OK

    # ---- copy-on-write
    def fork(self, dst: int, src: int) -> int:
        """dst shares every block of src, the partly filled last one included (parallel sampling)."""
        if src not in self.tables or src in self.swapped or dst in self.tables or dst == src:
            return E_INVALID
        for b in self.tables[src]:
            self.ref[b] += 1
        self.tables[dst] = list(self.tables[src])
        self.lens[dst] = self.lens[src]
        return OK

    def cow(self, seq: int, num_new: int = 1):
        """(status, src, dst) for a step about to write seq's last num_new positions (called after grow).

        The written positions are [len - num_new, len). If one of the blocks
        holding them is also named by another table (ref_count > 1), the first
        such block in table order is replaced, in seq's table only, by a block
        off the free list: the shared block loses one reference, the new one has
        ref_count 1, and (OK, shared block, new block) names the copy the
        caller makes before the step writes. (OK, -1, -1) when every such block
        is already seq's alone; (E_NOMEM, -1, -1) with nothing changed when no
        block is free. Several shared blocks take one call each."""
        if seq not in self.tables or seq in self.swapped:
            return E_INVALID, -1, -1
        n = self.lens[seq]
        if num_new < 0 or num_new > n:
            return E_INVALID, -1, -1
        t = self.tables[seq]
        written = range((n - num_new) // self.block_size, (n - 1) // self.block_size + 1) if num_new else ()
        shared = [i for i in written if self.ref[t[i]] > 1]
        if not shared:
            return OK, -1, -1
        if not self.free:
            return E_NOMEM, -1, -1
        i = shared[0]
        b = self.free.pop()
        self.ref[b] = 1
        old = t[i]
        self.ref[old] -= 1
        t[i] = b
        return OK, old, b

    # ---- swap
    def swap_out(self, seq: int):
        """(status, blocks): the blocks to copy to host, in table order; they are released."""
        if seq not in self.tables or seq in self.swapped:
            return E_INVALID, None
        blocks = self.tables[seq]
        for b in blocks:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)
        self.tables[seq] = []
        self.swapped.add(seq)
        return OK, list(blocks)

    def swap_in(self, seq: int):
        """(status, blocks): fresh blocks for the host copy to return to, in table order."""
        if seq not in self.swapped:
            return E_INVALID, None
        need = self.blocks_needed(self.lens[seq])
        if need > len(self.free):
            return E_NOMEM, None
        blocks = []
        for _ in range(need):
            b = self.free.pop()
            self.ref[b] = 1
            blocks.append(b)
        self.tables[seq] = blocks
        self.swapped.discard(seq)
        return OK, list(blocks)

    # ---- prefix cache
    def prefix_register(self, seq: int, hashes) -> tuple:
        """Cache seq's leading full blocks under their chained hashes. (status, newly cached). A block
        already cached under another hash is left as it is."""
        if seq not in self.tables or seq in self.swapped or len(hashes) * self.block_size > self.lens[seq]:
            return E_INVALID, 0
        self.clock += 1
        new = 0
        for i, h in enumerate(hashes):
            h = int(h)
            if h in self.cache:
                self.cache[h][1] = self.clock
                continue
            b = self.tables[seq][i]
            if b in self.cached_blocks:
                continue
            self.cache[h] = [b, self.clock, i]
            self.cached_blocks.add(b)
            self.ref[b] += 1
            new += 1
        return OK, new

    def prefix_match(self, hashes) -> int:
        n = 0
        for h in hashes:
            if int(h) not in self.cache:
                break
            n += 1
        return n

    def attach_prefix(self, seq: int, hashes) -> tuple:
        """Start seq on the cached blocks of its longest cached prefix. (status, blocks attached)."""
        if seq in self.tables:
            return E_INVALID, 0
        n = self.prefix_match(hashes)
        self.clock += 1
        table = []
        for h in hashes[:n]:
            e = self.cache[int(h)]
            e[1] = self.clock
            self.ref[e[0]] += 1
            table.append(e[0])
        self.tables[seq] = table
        self.lens[seq] = n * self.block_size
        return OK, n

    def prefix_evict(self, max_blocks: int) -> int:
        """Evict up to max_blocks entries that only the cache references; they return to the free list."""
        cand = sorted((e[1], -e[2], e[0], h) for h, e in self.cache.items() if self.ref[e[0]] == 1)
        n = 0
        for _, _, b, h in cand[:max(0, max_blocks)]:
            del self.cache[h]
            self.cached_blocks.discard(b)
            self.ref[b] = 0
            self.free.append(b)
            n += 1
        return n

    def free_blocks(self) -> int:
        return len(self.free)

    def build_step(self, seqs, q_lens, max_blocks: int):
        """Step metadata: (status, tables, ctx_lens, slots, q_start_loc).

        Row i's new tokens are its last q_lens[i] positions; each must land in
        a block this sequence owns alone (ref_count 1)."""
        tables = [[-1] * max_blocks for _ in seqs]
        ctx, slots, qstart = [], [], [0]
        for i, (s, q) in enumerate(zip(seqs, q_lens)):
            if s not in self.tables or s in self.swapped or q < 1 or q > self.lens[s]:
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
