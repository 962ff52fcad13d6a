"""libpkv's C ABI on the host (no GPU): exported symbols, pool arithmetic,
argument validation, and the ref-counted block manager against the oracle's
restatement (oracle/blockmgr.py)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from oracle import blockmgr

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_cache_scatter_gb300 import build
    build.build()
    import paged_kv_cache_scatter_gb300 as pkv
    pkv.load()
    return pkv


def _header_functions():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol(pkv):
    names = _header_functions()
    assert len(names) >= 20
    lib = pkv.load()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing
    assert set(names) == set(pkv.SIGNATURES), "binding and header disagree"


def test_pool_bytes_matches_page_ledger(pkv):
    assert pkv.Pool.bytes_needed(7152) == 7152 * 8388608 == 59995324416
    assert pkv.Pool.bytes_needed(1) == oracle.bytes_per_block(oracle.geom(1, 32, 32))
    assert pkv.Pool.bytes_needed(64, num_layers=1) == 64 * 262144
    bad = pkv.pkv_pool_desc(10, 32, 32, 64, 16, 0, 0, None, 0, None)
    assert pkv.load().pkv_pool_bytes(ctypes.byref(bad)) == 0


@pytest.mark.parametrize("field,value", [("head_dim", 64), ("block_size", 32), ("dtype", 2), ("num_blocks", 0),
                                         ("partition_tokens", 100), ("partition_tokens", 4096), ("num_heads", 0),
                                         ("num_q_heads", 6), ("num_q_heads", 2), ("num_q_heads", 2048)])
def test_pool_create_refuses_bad_descriptor(pkv, field, value):
    d = pkv.pkv_pool_desc(16, 2, 4, 128, 16, 0, 0, None, 0, None)
    setattr(d, field, value)
    h = ctypes.c_void_p()
    assert pkv.load().pkv_pool_create(ctypes.byref(d), ctypes.byref(h)) == pkv.PKV_E_INVALID
    assert pkv.load().pkv_last_error_string()


def test_partition_limit_depends_on_the_decode_kernel(pkv):
    # one-head FP16 pools: up to 2,048 tokens per partition; grouped-head and 8-bit pools: up to 4,096
    assert pkv.Pool(None, 64, num_heads=32, partition_tokens=2048).handle
    for kw in ({"num_heads": 8, "num_q_heads": 32}, {"num_heads": 32, "dtype": "int8"}):
        assert pkv.Pool(None, 64, partition_tokens=4096, **kw).handle
        with pytest.raises(pkv.PkvError):
            pkv.Pool(None, 64, partition_tokens=4160, **kw)
    with pytest.raises(pkv.PkvError):
        pkv.Pool(None, 64, num_heads=32, partition_tokens=2112)


def test_grouped_query_pool_ledger_and_workspace(pkv):
    # "Inference Infrastructure" (seeitflow), KV cache arithmetic: 8 K/V heads x 128 dims x 2 (K and V)
    # x 2 bytes x 32 layers = 131,072 B per token, 2,097,152 B per 16-token block.
    assert pkv.Pool.bytes_needed(1, num_heads=8) == 16 * 131072 == oracle.bytes_per_block(oracle.geom(1, 32, 8))
    gqa = pkv.Pool(None, 64, num_heads=8, num_q_heads=32)
    mha = pkv.Pool(None, 64, num_heads=32)
    mqa = pkv.Pool(None, 64, num_heads=1, num_q_heads=32)
    # split-K partials are per query head: the workspace follows num_q_heads, not the K/V heads
    for rows, width in [(32, 300), (5, 17), (1, 4)]:
        assert gqa.decode_workspace_bytes(rows, width) == mha.decode_workspace_bytes(rows, width)
        assert mqa.decode_workspace_bytes(rows, width) == mha.decode_workspace_bytes(rows, width)
    assert pkv.Pool(None, 64, num_heads=8, num_q_heads=8).decode_workspace_bytes(32, 300) < \
        gqa.decode_workspace_bytes(32, 300)


def test_int8_pool_bytes_and_refusals(pkv):
    # 8-bit tiles: 16 x 128 codes + 16 float32 scales = 2,112 B; the oracle's own ledger agrees
    for n, L, H in [(7152, 32, 32), (64, 1, 32), (10, 3, 8)]:
        got = pkv.Pool.bytes_needed(n, num_layers=L, num_heads=H, dtype="int8")
        assert got == n * L * 2 * H * 2112 == oracle.pool_bytes(oracle.geom(n, L, H, dtype=oracle.INT8))
    assert pkv.Pool.bytes_needed(1, dtype="int8") * 2 < pkv.Pool.bytes_needed(1) * 1.04
    # grouped query heads work over an 8-bit pool too; the workspace follows the query heads
    p = pkv.Pool(None, 64, num_heads=8, num_q_heads=32, dtype="int8")
    assert p.decode_workspace_bytes(32, 300) == pkv.Pool(None, 64, num_heads=32).decode_workspace_bytes(32, 300)


def test_block_hashes_match_the_oracle(pkv):
    rng = np.random.default_rng(7)
    for n in [0, 15, 16, 17, 160, 1203]:
        t = rng.integers(-2**31, 2**31 - 1, n, dtype=np.int64).astype(np.int32)
        assert np.array_equal(pkv.block_hashes(t), oracle.block_hashes(t))


@pytest.mark.parametrize("seed", range(6))
def test_fork_cow_swap_and_prefix_cache_match_the_oracle(pkv, seed):
    # the library's block manager against the oracle's restatement, operation by operation
    rng = np.random.default_rng(100 + seed)
    N = 40
    order = rng.permutation(N)
    p = pkv.Pool(None, N, num_layers=1, free_order=order)
    bm = blockmgr.BlockManager(N, free_order=order)
    seqs = list(range(8))
    toks = {s: rng.integers(0, 7, 1000).astype(np.int32) for s in seqs}
    for _ in range(600):
        op = int(rng.integers(0, 10))
        s = int(rng.choice(seqs))
        if op <= 1:
            n = bm.lens.get(s, 0) + int(rng.integers(0, 40))
            assert p.seq_grow(s, n) == bm.grow(s, n)
        elif op == 2:
            assert p.seq_free(s) == bm.free_seq(s)
        elif op == 3:
            d = int(rng.choice(seqs))
            assert p.seq_fork(d, s) == bm.fork(d, s)
            if d in bm.tables:
                toks[d] = toks[s].copy()
        elif op == 4:
            k = int(rng.integers(-1, bm.lens.get(s, 0) + 2))
            assert p.seq_cow(s, k) == bm.cow(s, k)
        elif op == 5:
            st, blocks = p.seq_swap_out(s)
            st2, blocks2 = bm.swap_out(s)
            assert st == st2 and (st != 0 or list(blocks) == blocks2)
        elif op == 6:
            st, blocks = p.seq_swap_in(s)
            st2, blocks2 = bm.swap_in(s)
            assert st == st2 and (st != 0 or list(blocks) == blocks2)
        elif op == 7 and s in bm.tables and s not in bm.swapped:
            h = oracle.block_hashes(toks[s][:bm.lens[s] // 16 * 16])
            assert p.prefix_register(s, h) == bm.prefix_register(s, h)
        elif op == 8:
            h = oracle.block_hashes(toks[s][:int(rng.integers(0, 300))])
            assert p.prefix_match(h) == bm.prefix_match(h)
            if s not in bm.tables:
                assert p.seq_attach_prefix(s, h) == bm.attach_prefix(s, h)
        else:
            k = int(rng.integers(0, 3))
            assert p.prefix_evict(k) == bm.prefix_evict(k)
        _compare(p, bm, seqs)
        assert p.prefix_cached_blocks() == len(bm.cache)
    # swapped sequences refuse growth and steps; freeing everything returns every block
    for s in seqs:
        assert p.seq_free(s) == bm.free_seq(s)
    assert p.prefix_evict(N) == bm.prefix_evict(N)
    assert p.free_blocks() == N == bm.free_blocks()


# the hand-worked copy-on-write cases of tests/test_blockmgr_pins.py, through the C ABI
@pytest.mark.parametrize("n, src_table, grown, pair, after, slot", [
    (15, [0], [0], (0, 1), [1], 31), (16, [0], [0, 1], (-1, -1), [0, 1], 16), (17, [0, 1], [0, 1], (1, 2), [0, 2], 33),
    (47, [0, 1, 2], [0, 1, 2], (2, 3), [0, 1, 3], 63), (48, [0, 1, 2], [0, 1, 2, 3], (-1, -1), [0, 1, 2, 3], 48)])
def test_cow_at_fork_lengths(pkv, n, src_table, grown, pair, after, slot):
    p = pkv.Pool(None, 10, num_layers=1)
    assert p.seq_grow(0, n) == pkv.PKV_OK and list(p.block_table(0)) == src_table
    assert p.seq_fork(1, 0) == pkv.PKV_OK and p.seq_grow(1, n + 1) == pkv.PKV_OK
    assert list(p.block_table(1)) == grown
    assert p.build_step([1], [1], 8)[0] == (pkv.PKV_OK if pair == (-1, -1) else pkv.PKV_E_SHARED)
    assert p.seq_cow(1, 1) == (pkv.PKV_OK, *pair)
    assert list(p.block_table(1)) == after and p.seq_cow(1, 1) == (pkv.PKV_OK, -1, -1)
    st, _, ctx, slots, _ = p.build_step([1], [1], 8)
    assert st == pkv.PKV_OK and list(ctx) == [n + 1] and list(slots) == [slot]
    assert p.seq_grow(0, n + 1) == pkv.PKV_OK and p.seq_cow(0, 1) == (pkv.PKV_OK, -1, -1)
    assert p.seq_cow(1, n + 2)[0] == pkv.PKV_E_INVALID and p.seq_cow(1, -1)[0] == pkv.PKV_E_INVALID


def test_cow_rewrite_of_shared_prefix_one_block_per_call(pkv):
    p = pkv.Pool(None, 10, num_layers=1)
    assert p.seq_grow(0, 48) == pkv.PKV_OK and p.seq_share_prefix(1, 0, 3) == pkv.PKV_OK
    assert p.seq_cow(1, 17) == (pkv.PKV_OK, 1, 3)
    assert p.seq_cow(1, 17) == (pkv.PKV_OK, 2, 4)
    assert p.seq_cow(1, 17) == (pkv.PKV_OK, -1, -1)
    assert list(p.block_table(1)) == [0, 3, 4] and [p.ref_count(b) for b in range(5)] == [2, 1, 1, 1, 1]


def test_prefix_evict_order_by_hand(pkv):
    # least recently used first, deeper chain positions first among equals: blocks 2, 1, 4, 3, 0
    p = pkv.Pool(None, 8, num_layers=1)
    rng = np.random.default_rng(0)
    a = pkv.block_hashes(rng.integers(0, 1000, 48).astype(np.int32))
    b = pkv.block_hashes(rng.integers(0, 1000, 32).astype(np.int32))
    assert p.seq_grow(0, 48) == pkv.PKV_OK and p.prefix_register(0, a) == (pkv.PKV_OK, 3)
    assert p.seq_grow(1, 32) == pkv.PKV_OK and p.prefix_register(1, b) == (pkv.PKV_OK, 2)
    assert p.seq_free(0) == pkv.PKV_OK and p.seq_free(1) == pkv.PKV_OK
    assert p.seq_attach_prefix(2, a[:1]) == (pkv.PKV_OK, 1) and p.seq_free(2) == pkv.PKV_OK
    order = []
    for _ in range(5):
        left = {x for x in range(5) if p.ref_count(x) == 1}
        assert p.prefix_evict(1) == 1
        gone = left - {x for x in range(5) if p.ref_count(x) == 1}
        assert len(gone) == 1
        order += list(gone)
    assert order == [2, 1, 4, 3, 0]
    assert p.seq_grow(3, 16) == pkv.PKV_OK and list(p.block_table(3)) == [0]   # evicted last, reused first


def test_swap_out_capacity_and_state_rules(pkv):
    p = pkv.Pool(None, 8, num_layers=1)
    assert p.seq_grow(0, 40) == pkv.PKV_OK
    lib = pkv.load()
    n = ctypes.c_int64()
    small = np.zeros(2, np.int32)
    assert lib.pkv_seq_swap_out(p.handle, 0, small.ctypes.data, 2, ctypes.byref(n)) == pkv.PKV_E_INVALID
    assert n.value == 3 and p.free_blocks() == 5          # refused: nothing changed
    st, blocks = p.seq_swap_out(0)
    assert st == pkv.PKV_OK and len(blocks) == 3 and p.free_blocks() == 8 and p.seq_len(0) == 40
    assert p.seq_grow(0, 41) == pkv.PKV_E_INVALID
    assert p.build_step([0], [1], 4)[0] == pkv.PKV_E_INVALID
    assert p.seq_swap_out(0)[0] == pkv.PKV_E_INVALID
    st, blocks = p.seq_swap_in(0)
    assert st == pkv.PKV_OK and len(blocks) == 3 and p.free_blocks() == 5


def test_free_order_must_be_a_permutation(pkv):
    with pytest.raises(pkv.PkvError):
        pkv.Pool(None, 4, num_layers=1, free_order=[0, 1, 1, 2])
    p = pkv.Pool(None, 4, num_layers=1, free_order=[3, 0, 2, 1])
    assert p.seq_grow(0, 40) == pkv.PKV_OK
    assert list(p.block_table(0)) == [3, 0, 2]


def test_host_only_pool_refuses_kernel_calls(pkv):
    p = pkv.Pool(None, 8, num_layers=1)
    lib = pkv.load()
    assert lib.pkv_kv_append(p.handle, 0, 16, 16, 8, 1, None) == pkv.PKV_E_INVALID
    assert lib.pkv_decode_attn(p.handle, 0, 16, 16, 1, 16, 1, 0.1, 16, None, 0, None) == pkv.PKV_E_INVALID
    assert lib.pkv_get_status(p.handle, None, None) == pkv.PKV_E_INVALID


def _compare(p, bm, seqs):
    assert p.free_blocks() == bm.free_blocks()
    for b in range(bm.num_blocks):
        assert p.ref_count(b) == bm.ref[b]
    for s in seqs:
        if s in bm.tables:
            assert list(p.block_table(s)) == bm.tables[s]
            assert p.seq_len(s) == bm.lens[s]
        else:
            assert p.seq_len(s) == -1


@pytest.mark.parametrize("seed", range(6))
def test_block_manager_matches_oracle_under_random_ops(pkv, seed):
    rng = np.random.default_rng(seed)
    N = 48
    order = rng.permutation(N)
    p = pkv.Pool(None, N, num_layers=2, free_order=order)
    bm = blockmgr.BlockManager(N, free_order=order)
    seqs = list(range(8))
    for _ in range(300):
        op = rng.integers(0, 5)
        s = int(rng.choice(seqs))
        if op <= 1:
            n = int(rng.integers(0, 200))
            assert p.seq_grow(s, n) == bm.grow(s, n)
        elif op == 2:
            src = int(rng.choice(seqs))
            nb = int(rng.integers(0, 6))
            assert p.seq_share_prefix(s, src, nb) == bm.share_prefix(s, src, nb)
        elif op == 3:
            assert p.seq_free(s) == bm.free_seq(s)
        else:
            live = [x for x in seqs if x in bm.tables]
            if not live:
                continue
            k = int(rng.integers(1, len(live) + 1))
            rows = [int(x) for x in rng.choice(live, k, replace=False)]
            qls = [int(rng.integers(1, max(2, bm.lens[r] + 1))) if bm.lens[r] > 0 else 1 for r in rows]
            want = bm.build_step(rows, qls, 16)
            got = p.build_step(rows, qls, 16)
            assert got[0] == want[0]
            if want[0] == blockmgr.OK:
                assert np.array_equal(got[1], np.array(want[1], np.int32))
                assert list(got[2]) == want[2]
                assert list(got[3]) == want[3]
                assert list(got[4]) == want[4]
                # slots agree with the oracle's slot function
                rot = np.repeat(np.arange(len(rows)), qls)
                pos = np.concatenate([np.arange(c - q, c) for c, q in zip(want[2], qls)])
                assert np.array_equal(got[3], oracle.slots(got[1], rot, pos))
        _compare(p, bm, seqs)


def test_soak_returns_every_block_to_the_free_list(pkv):
    # "llm-inference-batching", Cancellation and memory: after a soak the free list is back at 7,152.
    rng = np.random.default_rng(0)
    p = pkv.Pool(None, 7152, free_order=rng.permutation(7152))
    live = {}
    nxt = 0
    for step in range(400):
        # join
        while len(live) < 32:
            n = int(np.clip(rng.lognormal(6.5, 1.0), 50, 8000))
            if p.seq_grow(nxt, n) == pkv.PKV_E_NOMEM:
                break
            live[nxt] = int(rng.integers(1, 300))
            nxt += 1
        # decode one token per row; cancel ~2% per step; finish when budget is spent
        for s in list(live):
            if rng.random() < 0.02 or live[s] == 0:
                assert p.seq_free(s) == pkv.PKV_OK
                del live[s]
                continue
            st = p.seq_grow(s, p.seq_len(s) + 1)
            if st == pkv.PKV_E_NOMEM:           # preempt the row
                assert p.seq_free(s) == pkv.PKV_OK
                del live[s]
                continue
            live[s] -= 1
    for s in list(live):
        assert p.seq_free(s) == pkv.PKV_OK
    assert p.free_blocks() == 7152
    assert all(p.ref_count(b) == 0 for b in range(0, 7152, 97))


def test_build_step_refuses_writes_into_shared_blocks(pkv):
    p = pkv.Pool(None, 64, num_layers=1)
    assert p.seq_grow(0, 40) == pkv.PKV_OK
    assert p.seq_share_prefix(1, 0, 2) == pkv.PKV_OK
    assert p.ref_count(int(p.block_table(0)[0])) == 2
    st = p.build_step([1], [1], 8)[0]
    assert st == pkv.PKV_E_SHARED          # the last position of seq 1 is inside a shared block
    assert p.seq_grow(1, 33) == pkv.PKV_OK  # a private block for the new token
    st, tables, ctx, slots, qs = p.build_step([1, 0], [1, 1], 8)
    assert st == pkv.PKV_OK and list(ctx) == [33, 40] and list(qs) == [0, 1, 2]
    assert slots[0] // 16 == tables[0][2] and slots[0] % 16 == 0
    assert p.seq_share_prefix(2, 0, 3) == pkv.PKV_E_INVALID   # block 2 of seq 0 is not full
