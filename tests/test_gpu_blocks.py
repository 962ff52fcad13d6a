"""GPU parity of whole-block copies (copy-on-write), swap to host memory and back, and the
prefix cache used end to end, against the oracle.

Block copies and swaps must be bit-exact (whole blocks, every layer). A
sequence that was swapped out and back in, or that diverged from a fork
through copy-on-write, or that was started on cached prefix blocks, must
attend exactly as the oracle does over the same pool state.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return G.lib()


def _bytes(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy().reshape(-1).copy()


def _pools(N, L, H):
    return [("fp16", G.device_pool(N, L, H, seed=3), oracle.geom(N, L, H)),
            ("int8", G.device_pool_i8(N, L, H, seed=3), oracle.geom(N, L, H, dtype=oracle.INT8))]


@pytest.mark.parametrize("kind", [0, 1])
def test_copy_blocks_bit_exact(pkv, kind):
    N, L, H = 20, 3, 8
    dtype, pool, g = _pools(N, L, H)[kind]
    p = pkv.Pool(pool, N, num_layers=L, num_heads=H, dtype=dtype)
    host = _bytes(pool)
    pairs = np.array([[3, 7], [0, 11], [5, 2], [19, 4], [18, 18]], np.int32)
    p.copy_blocks(torch.from_numpy(pairs).cuda())
    assert p.get_status() == (pkv.PKV_OK, 0)
    hv = host.view(np.uint16) if dtype == "fp16" else host
    assert oracle.copy_blocks(hv, g, pairs) == -1
    assert np.array_equal(_bytes(pool), host)
    # an out-of-pool block: that pair is skipped and flagged, the others still copy
    p.copy_blocks(torch.tensor([[1, 9], [2, N]], dtype=torch.int32, device="cuda"))
    st, flags = p.get_status()
    assert st == pkv.PKV_E_DEVICE and flags & pkv.PKV_DEV_BAD_BLOCK
    assert oracle.copy_blocks(hv, g, np.array([[1, 9]], np.int32)) == -1
    assert np.array_equal(_bytes(pool), host)


@pytest.mark.parametrize("kind", [0, 1])
def test_swap_out_and_in_bit_exact(pkv, kind):
    N, L, H = 24, 2, 8
    dtype, pool, g = _pools(N, L, H)[kind]
    p = pkv.Pool(pool, N, num_layers=L, num_heads=H, dtype=dtype)
    host_pool = _bytes(pool)
    hv = host_pool.view(np.uint16) if dtype == "fp16" else host_pool
    bb = oracle.bytes_per_block(g)
    blocks = np.array([17, 3, 3, 0, 23, 9], np.int32)
    buf = torch.empty(len(blocks) * bb, dtype=torch.uint8).pin_memory()
    p.swap_blocks_out(torch.from_numpy(blocks).cuda(), buf)
    torch.cuda.synchronize()
    assert p.get_status() == (pkv.PKV_OK, 0)
    assert np.array_equal(buf.numpy(), oracle.swap_out(hv, g, blocks))
    dst = np.array([1, 2, 4, 5, 6, 8], np.int32)
    p.swap_blocks_in(torch.from_numpy(dst).cuda(), buf)
    assert p.get_status() == (pkv.PKV_OK, 0)
    assert oracle.swap_in(hv, g, dst, buf.numpy()) == -1
    assert np.array_equal(_bytes(pool), host_pool)
    with pytest.raises(pkv.PkvError):                       # pageable memory is refused
        p.swap_blocks_out(torch.from_numpy(blocks).cuda(), torch.empty(len(blocks) * bb, dtype=torch.uint8))


def _decode(pkv, p, layer, q, tables, ctx):
    out = torch.empty_like(q)
    ws = torch.empty(max(p.decode_workspace_bytes(q.shape[0], tables.shape[1]), 256), dtype=torch.uint8,
                     device="cuda")
    p.decode_attn(layer, q, tables, ctx, G.SCALE, out, ws)
    assert p.get_status() == (pkv.PKV_OK, 0)
    return out


def _table(p, s, width):
    t = np.full((1, width), -1, np.int32)
    b = p.block_table(s)
    t[0, :len(b)] = b
    return torch.from_numpy(t).cuda()


def test_decode_unchanged_after_swap_out_and_in(pkv):
    # the block manager picks new blocks on swap-in; attention over the restored sequence is bit-identical
    N, L, H = 64, 2, 32
    pool = G.device_pool(N, L, H, seed=5)
    p = pkv.Pool(pool, N, num_layers=L, num_heads=H)
    assert p.seq_grow(0, 300) == pkv.PKV_OK and p.seq_grow(1, 200) == pkv.PKV_OK
    q = workloads.normal_fp16((1, H, 128), 6).cuda()
    ctx = torch.tensor([300], dtype=torch.int32, device="cuda")
    before = [_decode(pkv, p, l, q, _table(p, 0, 32), ctx) for l in range(L)]
    st, out_blocks = p.seq_swap_out(0)
    assert st == pkv.PKV_OK
    bb = pkv.Pool.bytes_needed(1, L, H)
    buf = torch.empty(len(out_blocks) * bb, dtype=torch.uint8).pin_memory()
    p.swap_blocks_out(torch.from_numpy(out_blocks).cuda(), buf)
    assert p.seq_grow(2, 16 * 20) == pkv.PKV_OK              # another sequence takes the released blocks
    pool[torch.from_numpy(p.block_table(2).astype(np.int64)).cuda()] = 0   # and overwrites them
    st, in_blocks = p.seq_swap_in(0)
    assert st == pkv.PKV_OK and not np.array_equal(in_blocks, out_blocks)
    p.swap_blocks_in(torch.from_numpy(in_blocks).cuda(), buf)
    after = [_decode(pkv, p, l, q, _table(p, 0, 32), ctx) for l in range(L)]
    for a, b in zip(before, after):
        assert torch.equal(a, b)


@pytest.mark.parametrize("n", [15, 40, 47, 48])
def test_fork_copy_on_write_then_diverge(pkv, n):
    # parallel sampling: a fork shares every block, the partly filled last one included; before each
    # branch's next token the block manager hands the writer a private copy of a shared block the token
    # lands in (none when the token opens a new block: n = 48), the device copies it, and the two branches
    # diverge. n = 47: the token completes the shared block.
    N, L, H = 32, 1, 32
    pool = G.device_pool(N, L, H, seed=7)
    host = G.to_bits(pool).reshape(pool.shape).copy()
    g = oracle.geom(N, L, H)
    p = pkv.Pool(pool, N, num_layers=L, num_heads=H)
    assert p.seq_grow(0, n) == pkv.PKV_OK
    assert p.seq_fork(1, 0) == pkv.PKV_OK
    for s in (0, 1):
        assert p.seq_grow(s, n + 1) == pkv.PKV_OK
    lands_in_shared = n % 16 != 0
    assert p.build_step([1], [1], 4)[0] == (pkv.PKV_E_SHARED if lands_in_shared else pkv.PKV_OK)
    pairs = []
    for s in (1, 0):
        st, src, dst = p.seq_cow(s, 1)
        assert st == pkv.PKV_OK
        if src >= 0:
            pairs.append((src, dst))
    assert len(pairs) == (1 if lands_in_shared else 0)     # the second writer finds the block its own
    if pairs:
        pr = np.array(pairs, np.int32)
        p.copy_blocks(torch.from_numpy(pr).cuda())
        assert oracle.copy_blocks(host, g, pr) == -1
    st, tables, ctx, slots, qs = p.build_step([0, 1], [1, 1], 4)
    assert st == pkv.PKV_OK and slots[0] != slots[1]
    k = workloads.normal_fp16((2, H, 128), 8).cuda()
    v = workloads.normal_fp16((2, H, 128), 9).cuda()
    q = workloads.normal_fp16((2, H, 128), 10).cuda()
    p.kv_append(0, k, v, torch.from_numpy(slots).cuda())
    assert oracle.kv_append(host, g, 0, G.to_bits(k), G.to_bits(v), slots) == -1
    out = _decode(pkv, p, 0, q, torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda())
    ref, _ = oracle.decode_attn(host, g, 0, G.to_bits(q), tables, ctx, G.SCALE)
    G.assert_close(out, ref, "forked rows after copy-on-write")
    assert np.array_equal(G.to_bits(pool).reshape(pool.shape), host)
    assert not torch.equal(out[0], out[1])


def test_prefix_cache_prefill_only_the_suffix(pkv):
    # request A prefills its prompt and caches its full blocks; request B with the same system prompt starts
    # on those blocks and prefills only its own tokens; both attend as the oracle does
    N, L, H = 96, 1, 32
    pool = G.device_pool(N, L, H, seed=11)
    host = G.to_bits(pool).reshape(pool.shape).copy()
    g = oracle.geom(N, L, H)
    p = pkv.Pool(pool, N, num_layers=L, num_heads=H)
    rng = np.random.default_rng(11)
    system = rng.integers(0, 32000, 400).astype(np.int32)
    prompt_a = np.concatenate([system, rng.integers(0, 32000, 90).astype(np.int32)])
    prompt_b = np.concatenate([system, rng.integers(0, 32000, 130).astype(np.int32)])

    def prefill(seq, n_new, seed):
        st, tables, ctx, slots, qs = p.build_step([seq], [n_new], 40)
        assert st == pkv.PKV_OK
        k = workloads.normal_fp16((n_new, H, 128), seed).cuda()
        v = workloads.normal_fp16((n_new, H, 128), seed + 1).cuda()
        q = workloads.normal_fp16((n_new, H, 128), seed + 2).cuda()
        p.kv_append(0, k, v, torch.from_numpy(slots).cuda())
        out = torch.empty_like(q)
        p.prefill_attn(0, q, torch.from_numpy(qs).cuda(), torch.from_numpy(tables).cuda(),
                       torch.from_numpy(ctx).cuda(), n_new, G.SCALE, out)
        assert p.get_status() == (pkv.PKV_OK, 0)
        assert oracle.kv_append(host, g, 0, G.to_bits(k), G.to_bits(v), slots) == -1
        ref, _ = oracle.prefill_attn(host, g, 0, G.to_bits(q), qs, tables, ctx, G.SCALE)
        G.assert_close(out, ref, f"prefill of seq {seq}")

    assert p.seq_grow(0, len(prompt_a)) == pkv.PKV_OK
    prefill(0, len(prompt_a), 20)
    ha = pkv.block_hashes(prompt_a)
    assert np.array_equal(ha, oracle.block_hashes(prompt_a))
    assert p.prefix_register(0, ha) == (pkv.PKV_OK, len(prompt_a) // 16)
    hb = pkv.block_hashes(prompt_b)
    st, n = p.seq_attach_prefix(1, hb)
    assert st == pkv.PKV_OK and n == len(system) // 16      # the shared 400 tokens: 25 full blocks
    assert list(p.block_table(1)) == list(p.block_table(0))[:n]
    assert p.seq_grow(1, len(prompt_b)) == pkv.PKV_OK
    prefill(1, len(prompt_b) - 16 * n, 30)                   # only the 130 tokens past the cached blocks
    assert np.array_equal(G.to_bits(pool).reshape(pool.shape), host)
    assert p.seq_free(0) == pkv.PKV_OK and p.seq_free(1) == pkv.PKV_OK
    assert p.prefix_cached_blocks() == len(prompt_a) // 16
    assert p.prefix_evict(1000) == len(prompt_a) // 16 and p.free_blocks() == N
