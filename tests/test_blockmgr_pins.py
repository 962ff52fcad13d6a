"""Pins for the oracle's block manager (oracle/blockmgr.py), fixed by the pages' rules and worked by hand.

The pages fix the bookkeeping in words and small listings: ceil(tokens / 16)
blocks per sequence, blocks popped from the end of a free list and returned
to it ("continuous batching server", "The KV Cache Block Manager"), refusal
with no change when the list runs out ("Serving LLMs", "Paged KV memory"),
reference counts above 1 on shared blocks ("llm-inference-batching", the KV
pool listing), copy-on-write when a branch diverges ("The inference
engine", "Paging turns variable sequences into block tables"), and a cache
of full blocks keyed by chained hashes whose entries are evicted least
recently used first ("Serving LLMs", "Prefix caching"). The expected block
ids below are worked out from those rules with a pool whose free list hands
out 0, 1, 2, ... in order, not read back from the oracle.

tests/test_oracle_mutants.py runs this file against mutated copies of
oracle/blockmgr.py (the path arrives in PKV_ORACLE_BLOCKMGR) and checks that
each planted mistake fails a pin here.
"""
import importlib.util
import math
import os

import numpy as np
import pytest

import oracle


def _load_blockmgr():
    path = os.environ.get("PKV_ORACLE_BLOCKMGR")
    if not path:
        from oracle import blockmgr as m
        return m
    spec = importlib.util.spec_from_file_location("blockmgr_under_test", path)
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


blockmgr = _load_blockmgr()
OK, E_INVALID, E_NOMEM, E_SHARED = blockmgr.OK, blockmgr.E_INVALID, blockmgr.E_NOMEM, blockmgr.E_SHARED


def _state(bm):
    return list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()}, dict(bm.lens)


def test_blockmgr_page_example_lengths():
    bm = blockmgr.BlockManager(7152)
    for i, n in enumerate([17, 33, 65]):
        assert bm.grow(i, n) == blockmgr.OK
    assert 7152 - bm.free_blocks() == 10
    assert bm.grow(3, 600) == blockmgr.OK and len(bm.tables[3]) == 38
    assert bm.grow(4, 2300) == blockmgr.OK and len(bm.tables[4]) == 144


def test_blockmgr_grow_one_block_every_16_tokens():
    bm = blockmgr.BlockManager(64)
    for n in range(1, 200):
        assert bm.grow(0, n) == blockmgr.OK
        assert len(bm.tables[0]) == math.ceil(n / 16)


def test_blockmgr_nomem_changes_nothing():
    bm = blockmgr.BlockManager(8)
    assert bm.grow(0, 100) == blockmgr.OK           # 7 blocks
    before = (list(bm.free), list(bm.tables[0]), bm.lens[0])
    assert bm.grow(1, 40) == blockmgr.E_NOMEM
    assert bm.grow(0, 129) == blockmgr.E_NOMEM
    assert (list(bm.free), list(bm.tables[0]), bm.lens[0]) == before and 1 not in bm.tables


def test_blockmgr_shared_prefix_refcounts_and_soak_returns_all_blocks():
    bm = blockmgr.BlockManager(7152, free_order=np.random.default_rng(0).permutation(7152))
    assert bm.grow(0, 2000) == blockmgr.OK
    for s in range(1, 65):
        assert bm.share_prefix(s, 0, 125) == blockmgr.OK
        assert bm.grow(s, 2000 + s) == blockmgr.OK
    shared = bm.tables[0][:125]
    assert all(bm.ref[b] == 65 for b in shared)
    st, tables, ctx, slots, qs = bm.build_step(list(range(1, 65)), [1] * 64, 200)
    assert st == blockmgr.OK and len(slots) == 64
    assert all(s // 16 not in shared for s in slots)
    # a write into a shared block is refused
    assert bm.grow(99, 0) == blockmgr.OK
    assert bm.share_prefix(100, 0, 10) == blockmgr.OK
    assert bm.build_step([100], [1], 200)[0] == blockmgr.E_SHARED
    for s in list(bm.tables):
        assert bm.free_seq(s) == blockmgr.OK
    assert bm.free_blocks() == 7152 and all(r == 0 for r in bm.ref)


def test_blockmgr_lifo_reuse_and_invalid_calls():
    bm = blockmgr.BlockManager(10)
    assert bm.grow(0, 40) == blockmgr.OK
    assert bm.tables[0] == [0, 1, 2]
    assert bm.free_seq(0) == blockmgr.OK
    assert bm.grow(1, 16) == blockmgr.OK and bm.tables[1] == [2]
    assert bm.free_seq(7) == blockmgr.E_INVALID
    assert bm.grow(1, 3) == blockmgr.E_INVALID          # sequences only grow
    assert bm.share_prefix(2, 1, 2) == blockmgr.E_INVALID  # only full blocks that exist



def _page_prefill_with_cache(cache: set, tokens) -> int:
    """The page's lookup: count cached leading blocks until the first miss, then cache this prompt's blocks."""
    hit = 0
    hs = [int(x) for x in oracle.block_hashes(tokens)]
    for h in hs:
        if h not in cache:
            break
        hit += 16
    cache.update(hs)
    return hit


def test_prefix_cache_matches_the_pages_lookup():
    rng = np.random.default_rng(1)
    system = rng.integers(0, 32000, 1200).astype(np.int32)            # a shared 1,200-token system prompt
    bm = blockmgr.BlockManager(4000)
    page_cache: set = set()
    for r in range(20):
        user = rng.integers(0, 32000, int(rng.integers(1, 900))).astype(np.int32)
        prompt = np.concatenate([system, user]) if r % 4 else user
        hs = oracle.block_hashes(prompt)
        expect = _page_prefill_with_cache(page_cache, prompt)
        st, n = bm.attach_prefix(r, hs)
        assert st == blockmgr.OK and n * 16 == expect
        assert bm.grow(r, len(prompt)) == blockmgr.OK
        assert bm.prefix_register(r, hs)[0] == blockmgr.OK
    # a changed token near the start of the system prompt: nothing is served from the cache
    p = np.concatenate([system, [5, 6, 7]]).astype(np.int32)
    p[3] += 1
    assert bm.prefix_match(oracle.block_hashes(p)) == 0 == _page_prefill_with_cache(set(page_cache), p)
    assert bm.prefix_match(oracle.block_hashes(system)) == 1200 // 16



def test_blockmgr_nomem_leaves_state_unchanged_for_cow_and_swap_in():
    bm = blockmgr.BlockManager(4)
    assert bm.grow(0, 20) == blockmgr.OK and bm.fork(1, 0) == blockmgr.OK
    assert bm.grow(2, 32) == blockmgr.OK                  # pool full
    snap = (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()})
    assert bm.grow(1, 21) == blockmgr.OK            # position 20 falls in shared block 1
    snap = (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()})
    assert bm.cow(1, 1) == (blockmgr.E_NOMEM, -1, -1)
    assert snap == (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()})
    assert bm.swap_out(2)[0] == blockmgr.OK and bm.grow(3, 32) == blockmgr.OK
    snap = (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()})
    assert bm.swap_in(2) == (blockmgr.E_NOMEM, None)
    assert snap == (list(bm.free), list(bm.ref), {k: list(v) for k, v in bm.tables.items()})


def test_blockmgr_reference_counts_under_random_operations():
    # invariant: ref[b] = number of table entries naming b + 1 if b is cached; free list = blocks with ref 0
    rng = np.random.default_rng(3)
    N = 64
    bm = blockmgr.BlockManager(N, free_order=rng.permutation(N))
    toks = {}
    for step in range(3000):
        op = rng.integers(0, 9)
        s = int(rng.integers(0, 12))
        if op == 0:
            bm.grow(s, bm.lens.get(s, 0) + int(rng.integers(0, 40)))
        elif op == 1:
            bm.free_seq(s)
        elif op == 2:
            bm.fork(int(rng.integers(0, 12)), s)
        elif op == 3:
            if s in bm.lens:
                bm.cow(s, int(rng.integers(0, bm.lens[s] + 1)))
        elif op == 4:
            bm.swap_out(s)
        elif op == 5:
            bm.swap_in(s)
        elif op == 6 and s in bm.tables and s not in bm.swapped:
            n = bm.lens[s] // 16 * 16
            toks.setdefault(s, rng.integers(0, 9, 4000).astype(np.int32))
            bm.prefix_register(s, oracle.block_hashes(toks[s][:n]))
        elif op == 7 and s not in bm.tables:
            toks[s] = rng.integers(0, 9, 4000).astype(np.int32)
            bm.attach_prefix(s, oracle.block_hashes(toks[s][:int(rng.integers(0, 200))]))
        elif op == 8:
            bm.prefix_evict(int(rng.integers(0, 4)))
        count = [0] * N
        for t in bm.tables.values():
            for b in t:
                count[b] += 1
        for e in bm.cache.values():
            count[e[0]] += 1
        assert count == bm.ref
        assert sorted(bm.free) == [b for b in range(N) if bm.ref[b] == 0]
    for s in list(bm.tables):
        bm.free_seq(s)
    bm.prefix_evict(N)
    assert bm.free_blocks() == N and not bm.cache


# ------------------------------------------------------------------ copy-on-write
# Rule ("The inference engine" (wpnews), "Paging turns variable sequences into block tables"): a branch
# that is about to write into a block another branch still holds first gets its own copy of that block;
# blocks it does not write stay shared. A fork shares every block, the partly filled last one included.
# The call comes after grow, for the positions the coming step writes: [len - num_new, len).

# (fork length, the source's table, the branch's table after growing by one token, the (src, dst) copy
#  the branch needs, its table afterwards, the slot its new token gets)
FORK_CASES = [
    # 15 tokens: position 15 is the last slot of block 0, which both hold -> copy it into block 1
    (15, [0], [0], (0, 1), [1], 1 * 16 + 15),
    # 16 tokens: block 0 is full; position 16 opens block 1, which grow gave the branch alone -> no copy
    (16, [0], [0, 1], (-1, -1), [0, 1], 1 * 16 + 0),
    # 17 tokens: position 17 is the second slot of shared block 1 -> copy it into block 2
    (17, [0, 1], [0, 1], (1, 2), [0, 2], 2 * 16 + 1),
    # 47 tokens: position 47 completes shared block 2 -> copy it into block 3
    (47, [0, 1, 2], [0, 1, 2], (2, 3), [0, 1, 3], 3 * 16 + 15),
    # 48 tokens: blocks 0-2 are full; position 48 opens block 3, the branch's own -> no copy
    (48, [0, 1, 2], [0, 1, 2, 3], (-1, -1), [0, 1, 2, 3], 3 * 16 + 0),
]


@pytest.mark.parametrize("n, src_table, grown, pair, after, slot", FORK_CASES)
def test_cow_at_fork_lengths_by_hand(n, src_table, grown, pair, after, slot):
    bm = blockmgr.BlockManager(10)
    assert bm.grow(0, n) == OK and bm.tables[0] == src_table
    assert bm.fork(1, 0) == OK and bm.lens[1] == n
    assert all(bm.ref[b] == 2 for b in src_table)
    assert bm.grow(1, n + 1) == OK and bm.tables[1] == grown
    shared_write = pair != (-1, -1)
    assert bm.build_step([1], [1], 8)[0] == (E_SHARED if shared_write else OK)
    assert bm.cow(1, 1) == (OK, *pair)
    assert bm.tables[1] == after and bm.tables[0] == src_table
    if shared_write:
        assert bm.ref[pair[0]] == 1 and bm.ref[pair[1]] == 1
    assert bm.cow(1, 1) == (OK, -1, -1)                   # nothing left to copy
    st, _, ctx, slots, _ = bm.build_step([1], [1], 8)
    assert st == OK and ctx == [n + 1] and slots == [slot]
    # the source then takes its own next token: the block it kept is now its alone
    assert bm.grow(0, n + 1) == OK
    assert bm.cow(0, 1) == (OK, -1, -1)
    st, _, _, slots2, _ = bm.build_step([0, 1], [1, 1], 8)
    assert st == OK and slots2[1] == slot and slots2[0] != slot


def test_cow_multi_token_write_and_shared_prefix_rewrite():
    bm = blockmgr.BlockManager(10)
    # a fork at 40 whose branch then writes 20 tokens at once: positions 40..59 span shared block 2 and the
    # branch's new block 3; only block 2 is copied (into block 4)
    assert bm.grow(0, 40) == OK and bm.fork(1, 0) == OK
    assert bm.grow(1, 60) == OK and bm.tables[1] == [0, 1, 2, 3]
    assert bm.build_step([1], [20], 8)[0] == E_SHARED
    assert bm.cow(1, 20) == (OK, 2, 4)
    assert bm.cow(1, 20) == (OK, -1, -1)
    st, _, _, slots, _ = bm.build_step([1], [20], 8)
    assert st == OK and slots == [4 * 16 + p % 16 for p in range(40, 48)] + [3 * 16 + p % 16 for p in range(48, 60)]
    # a rewrite of the last 17 tokens of a shared 3-block prefix touches blocks 1 and 2: one copy per call,
    # in table order
    bm = blockmgr.BlockManager(10)
    assert bm.grow(0, 48) == OK and bm.share_prefix(1, 0, 3) == OK
    assert bm.cow(1, 17) == (OK, 1, 3)
    assert bm.cow(1, 17) == (OK, 2, 4)
    assert bm.cow(1, 17) == (OK, -1, -1)
    assert bm.tables[1] == [0, 3, 4] and [bm.ref[b] for b in range(5)] == [2, 1, 1, 1, 1]
    assert bm.build_step([1], [17], 8)[0] == OK
    assert bm.cow(1, 0) == (OK, -1, -1)                   # nothing written, nothing copied


def test_cow_refusals_change_nothing():
    bm = blockmgr.BlockManager(3)
    assert bm.grow(0, 20) == OK and bm.fork(1, 0) == OK and bm.grow(1, 21) == OK
    assert bm.grow(2, 1) == OK                             # pool full: 0, 1 shared, 2 for seq 2
    snap = _state(bm)
    assert bm.cow(1, 1) == (E_NOMEM, -1, -1)
    assert bm.cow(1, 22) == (E_INVALID, -1, -1)           # more new tokens than the sequence holds
    assert bm.cow(1, -1) == (E_INVALID, -1, -1)
    assert bm.cow(9, 1) == (E_INVALID, -1, -1)            # unknown sequence
    assert _state(bm) == snap
    assert bm.free_seq(2) == OK
    assert bm.cow(1, 1) == (OK, 1, 2)


def test_cow_then_build_step_never_refuses_under_random_operations():
    # after grow and the cow calls for a step's q tokens, build_step accepts the row; blocks the step does
    # not write stay shared
    rng = np.random.default_rng(5)
    for trial in range(60):
        bm = blockmgr.BlockManager(64, free_order=rng.permutation(64))
        assert bm.grow(0, int(rng.integers(1, 120))) == OK
        for s in range(1, 4):
            assert bm.fork(s, int(rng.integers(0, s))) == OK
        for s in range(4):
            q = int(rng.integers(1, 30))
            assert bm.grow(s, bm.lens[s] + q) == OK
            before = list(bm.tables[s])
            copies = []
            while True:
                st, a, b = bm.cow(s, q)
                assert st == OK
                if a < 0:
                    break
                copies.append((a, b))
            assert bm.build_step([s], [q], 16)[0] == OK
            n = bm.lens[s]
            written = set(range((n - q) // 16, (n - 1) // 16 + 1))
            after = bm.tables[s]
            assert len(after) == len(before)
            changed = [(b0, b1) for i, (b0, b1) in enumerate(zip(before, after)) if b0 != b1]
            assert all(before[i] == after[i] for i in range(len(before)) if i not in written)
            assert changed == copies                       # one copy per replaced block, in table order


def test_blockmgr_swap_scenario():
    bm = blockmgr.BlockManager(10)
    assert bm.grow(0, 40) == OK and bm.fork(1, 0) == OK and bm.grow(1, 41) == OK
    assert bm.cow(1, 1) == (OK, 2, 3)
    st, blocks = bm.swap_out(1)
    assert st == OK and blocks == [0, 1, 3]
    assert bm.ref[3] == 0 and bm.ref[0] == 1 and bm.free_blocks() == 7 and bm.lens[1] == 41
    assert bm.grow(1, 50) == E_INVALID and bm.build_step([1], [1], 4)[0] == E_INVALID
    assert bm.cow(1, 1) == (E_INVALID, -1, -1)
    st, blocks = bm.swap_in(1)
    assert st == OK and blocks == [3, 4, 5] and bm.tables[1] == blocks   # LIFO: 3 was freed last
    assert all(bm.ref[b] == 1 for b in blocks) and bm.free_blocks() == 4


# ------------------------------------------------------------------ prefix-cache eviction
# Reading of "Serving LLMs" (sreshtalluri), "Prefix caching" (LRU for its radix-tree variant): an entry may
# be evicted once only the cache references its block; least recently used (registered or attached) first;
# among entries used at the same time, deeper chain positions first (a chain's tail goes before its head).

def _lru_scenario():
    bm = blockmgr.BlockManager(8)
    rng = np.random.default_rng(0)
    a = oracle.block_hashes(rng.integers(0, 1000, 48).astype(np.int32))   # three blocks
    b = oracle.block_hashes(rng.integers(0, 1000, 32).astype(np.int32))   # two blocks
    assert bm.grow(0, 48) == OK and bm.tables[0] == [0, 1, 2]
    assert bm.prefix_register(0, a) == (OK, 3)           # time 1: a0->0 (depth 0), a1->1 (1), a2->2 (2)
    assert bm.grow(1, 32) == OK and bm.tables[1] == [3, 4]
    assert bm.prefix_register(1, b) == (OK, 2)           # time 2: b0->3 (0), b1->4 (1)
    assert bm.free_seq(0) == OK and bm.free_seq(1) == OK
    assert bm.attach_prefix(2, a[:1]) == (OK, 1)         # time 3: a0 used again
    assert bm.free_seq(2) == OK
    assert [bm.ref[x] for x in range(5)] == [1] * 5      # only the cache holds them
    return bm, a, b


def test_prefix_evict_least_recently_used_then_deepest_first():
    # time 1: a2 (depth 2), a1 (depth 1); time 2: b1, b0; time 3: a0 -> blocks 2, 1, 4, 3, 0
    bm, a, b = _lru_scenario()
    # the lookup walks the chain and stops at the first miss: a miss first hides every later hit
    assert bm.prefix_match(list(a)) == 3 and bm.prefix_match([int(b[0]) ^ 1] + list(a)) == 0
    order = []
    for _ in range(5):
        free_before = bm.free_blocks()
        assert bm.prefix_evict(1) == 1
        assert bm.free_blocks() == free_before + 1
        order.append(bm.free[-1])
        assert bm.ref[order[-1]] == 0
    assert order == [2, 1, 4, 3, 0]
    assert bm.prefix_evict(1) == 0 and not bm.cache


def test_prefix_evict_batches_skip_referenced_entries_and_return_blocks_lifo():
    bm, a, b = _lru_scenario()
    assert bm.attach_prefix(5, b) == (OK, 2)             # time 4: b0, b1 in use by seq 5 (ref 2)
    assert bm.prefix_evict(2) == 2                       # a2, a1 (b's entries are referenced)
    assert bm.free[-2:] == [2, 1]
    assert bm.prefix_match(a) == 1 and bm.prefix_match(b) == 2
    assert bm.prefix_evict(10) == 1                      # only a0 is unreferenced now
    assert bm.free[-1] == 0 and bm.prefix_match(a) == 0 and bm.prefix_match(b) == 2
    assert bm.grow(6, 16) == OK and bm.tables[6] == [0]   # the block evicted last is handed out first
    assert bm.free_seq(5) == OK
    assert bm.prefix_evict(10) == 2 and bm.free[-2:] == [4, 3]    # b1 (deeper) before b0, same time 4
    assert bm.prefix_evict(0) == 0 and bm.prefix_evict(-3) == 0
