"""GPU parity of kv_append and paged decode attention against the oracle.

All calls go through libpkv's C ABI. Inputs are seeded (workloads/); the
oracle sees host copies of the same bytes and never anything the CUDA path
produced. kv_append must match bit for bit (including untouched canary
rows); attention must satisfy |gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise.
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


def _decode(pkv, p, layer, q, tables_d, ctx_d):
    out = torch.full_like(q, float("nan"))
    ws = torch.empty(max(p.decode_workspace_bytes(q.shape[0], tables_d.shape[1]), 256), dtype=torch.uint8,
                     device="cuda")
    p.decode_attn(layer, q, tables_d, ctx_d, G.SCALE, out, ws)
    st, flags = p.get_status()
    assert st == pkv.PKV_OK and flags == 0, (st, flags)
    return out


# ------------------------------------------------------------------ kv_append

@pytest.mark.parametrize("layer,T", [(0, 1), (2, 37), (1, 300)])
def test_kv_append_bit_exact_and_canaries_untouched(pkv, layer, T):
    N, L, H = 40, 3, 32
    pool = G.device_pool(N, L, H, seed=1)
    host = G.to_bits(pool).reshape(pool.shape).copy()
    p = pkv.Pool(pool, N, num_layers=L, num_heads=H)
    rng = np.random.default_rng(T)
    slots = rng.choice(N * 16, T, replace=False).astype(np.int64)
    k = workloads.normal_fp16((T, H, 128), 11 + T).cuda()
    v = workloads.normal_fp16((T, H, 128), 12 + T).cuda()
    p.kv_append(layer, k, v, torch.from_numpy(slots).cuda())
    st, flags = p.get_status()
    assert st == pkv.PKV_OK and flags == 0
    g = oracle.geom(N, L, H)
    assert oracle.kv_append(host, g, layer, G.to_bits(k), G.to_bits(v), slots) == -1
    assert np.array_equal(G.to_bits(pool).reshape(pool.shape), host)


def test_kv_append_rejects_bad_slot_on_device(pkv):
    N, L, H = 8, 1, 4
    pool = G.device_pool(N, L, H, seed=2)
    before = G.to_bits(pool).copy()
    p = pkv.Pool(pool, N, num_layers=L, num_heads=H)
    k = torch.ones(2, H, 128, dtype=torch.float16, device="cuda")
    p.kv_append(0, k, k, torch.tensor([N * 16, -5], dtype=torch.int64, device="cuda"))
    st, flags = p.get_status()
    assert st == pkv.PKV_E_DEVICE and flags & pkv.PKV_DEV_BAD_SLOT
    assert np.array_equal(G.to_bits(pool), before)
    assert p.get_status() == (pkv.PKV_OK, 0)   # the flag was cleared and the context is fine


# ------------------------------------------------------------------ decode

def _run_decode_case(pkv, wl, partition=0, layers=(0,)):
    """Append each row's new token, then decode; compare with the oracle."""
    pool = G.device_pool(wl.num_blocks, wl.num_layers, wl.num_heads, seed=wl.seed)
    host = G.to_bits(pool).reshape(pool.shape).copy()
    p = pkv.Pool(pool, wl.num_blocks, num_layers=wl.num_layers, num_heads=wl.num_heads, partition_tokens=partition)
    tables_d, ctx_d, _, slots_d, slots = G.step_metadata(wl)
    g = oracle.geom(wl.num_blocks, wl.num_layers, wl.num_heads)
    errs = []
    for layer in layers:
        q, k, v = G.new_token_inputs(wl, layer)
        p.kv_append(layer, k, v, slots_d)
        out = _decode(pkv, p, layer, q, tables_d, ctx_d)
        assert oracle.kv_append(host, g, layer, G.to_bits(k), G.to_bits(v), slots) == -1
        ref64, _ = oracle.decode_attn(host, g, layer, G.to_bits(q), wl.block_tables, wl.ctx_lens, G.SCALE)
        errs.append(G.assert_close(out, ref64, f"{wl.name} layer {layer}"))
    assert np.array_equal(G.to_bits(pool).reshape(pool.shape), host), "pool differs from the oracle's after append"
    return errs


def test_tiny_decode_config(pkv):
    # 1 layer, 4 rows, contexts 17/50/100/255, 64-block permuted pool
    _run_decode_case(pkv, workloads.tiny_decode(0))


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("partition", [0, 64, 2048])
def test_random_ragged_decode(pkv, seed, partition):
    wl = workloads.random_step(seed, num_seqs=9, max_ctx=1500, num_blocks=900, num_layers=2)
    wl.ctx_lens[0] = 1                       # a row with only its new token
    wl.ctx_lens[1] = 16                      # exactly one full block
    _run_decode_case(pkv, wl, partition, layers=(1,))


@pytest.mark.parametrize("partition,ctxs", [(0, [1024, 1025, 1040, 1041, 2047, 2048, 2049, 3073]),
                                            (64, [64, 65, 80, 127, 128, 129, 1000, 3073])])
def test_decode_equal_partition_boundaries(pkv, partition, ctxs):
    # Contexts on and next to the partition bounds (0 = the library's 1,024): a row's keys go into the fewest
    # partitions of at most that many keys, of equal length in whole blocks, which must cover [0, ctx) once.
    wl = workloads.random_step(13, num_seqs=len(ctxs), max_ctx=3100, min_ctx=3100,
                               num_blocks=len(ctxs) * 194 + 8, num_layers=1)
    wl.ctx_lens[:] = ctxs
    _run_decode_case(pkv, wl, partition)


def test_decode_long_rows_many_partitions(pkv):
    wl = workloads.random_step(7, num_seqs=3, max_ctx=4200, min_ctx=3000, num_blocks=800, num_layers=1)
    _run_decode_case(pkv, wl, partition=64)


def test_one_hot_softmax_returns_value_row_exactly(pkv):
    N, L, H = 16, 1, 32
    ctx = 37
    pool = G.device_pool(N, L, H, seed=3)
    rng = np.random.default_rng(3)
    table = rng.permutation(N)[:3].astype(np.int32)
    q = workloads.normal_fp16((1, H, 128), 5).cuda()
    p = pkv.Pool(pool, N, num_layers=L, num_heads=H)
    for j in (0, 15, 16, 36):
        pos = np.arange(ctx)
        blk, off = table[pos // 16], pos % 16
        pool[torch.from_numpy(blk.astype(np.int64)).cuda(), 0, 0] = 0
        pool[int(blk[j]), 0, 0, :, int(off[j]), :] = (q[0].double() * 128).half()
        out = _decode(pkv, p, 0, q, torch.from_numpy(table[None]).cuda(), torch.tensor([ctx], dtype=torch.int32,
                                                                                         device="cuda"))
        vj = pool[int(blk[j]), 0, 1, :, int(off[j]), :]
        assert torch.equal(out[0], vj)


def test_batch_invariance(pkv):
    # "llm-inference-batching", Correctness: a request alone and in a mixed batch gives the same result.
    wl = workloads.random_step(11, num_seqs=12, max_ctx=2600, num_blocks=1200, num_layers=1)
    pool = G.device_pool(wl.num_blocks, 1, 32, seed=11)
    p = pkv.Pool(pool, wl.num_blocks, num_layers=1)
    tables_d, ctx_d, _, _, _ = G.step_metadata(wl)
    q, _, _ = G.new_token_inputs(wl, 0)
    together = _decode(pkv, p, 0, q, tables_d, ctx_d)
    for r in range(wl.num_seqs):
        alone = _decode(pkv, p, 0, q[r:r + 1].contiguous(), tables_d[r:r + 1].contiguous(), ctx_d[r:r + 1].contiguous())
        assert torch.equal(alone[0], together[r])


def test_physical_block_permutation_invariance(pkv):
    wl = workloads.random_step(12, num_seqs=6, max_ctx=1800, num_blocks=700, num_layers=1)
    pool = G.device_pool(wl.num_blocks, 1, 32, seed=12)
    p = pkv.Pool(pool, wl.num_blocks, num_layers=1)
    tables_d, ctx_d, _, _, _ = G.step_metadata(wl)
    q, _, _ = G.new_token_inputs(wl, 0)
    ref = _decode(pkv, p, 0, q, tables_d, ctx_d)
    perm = torch.from_numpy(np.random.default_rng(0).permutation(wl.num_blocks)).cuda()
    moved = torch.empty_like(pool)
    moved[perm] = pool
    p2 = pkv.Pool(moved, wl.num_blocks, num_layers=1)
    t2 = torch.where(tables_d >= 0, perm[tables_d.clamp(min=0).long()].int(), tables_d)
    got = _decode(pkv, p2, 0, q, t2, ctx_d)
    assert torch.equal(ref, got)


def test_marker_rows_read_only_their_blocks(pkv):
    # "llm-inference-batching", Correctness: no request's output shows another request's marker.
    N, H = 64, 32
    pool = torch.full(workloads.pool_shape(N, 1, H), 1000.0, dtype=torch.float16, device="cuda")
    pool[:, :, 0] = 0                                         # K = 0: uniform softmax
    shared = [40, 7, 22]
    nrows = 5
    priv_tokens = [1, 17, 30, 48, 5]
    tables = np.full((nrows, 8), -1, np.int32)
    cursor = 0
    free = [b for b in range(N) if b not in shared]
    for r in range(nrows):
        nb = -(-priv_tokens[r] // 16)
        mine = free[cursor:cursor + nb]
        cursor += nb
        tables[r, :3] = shared
        tables[r, 3:3 + nb] = mine
        pool[mine, :, 1] = float(r + 1) / 8
    pool[shared, :, 1] = -2.0
    ctx = np.array([48 + t for t in priv_tokens], np.int32)
    p = pkv.Pool(pool, N, num_layers=1)
    q = workloads.normal_fp16((nrows, H, 128), 9).cuda()
    out = _decode(pkv, p, 0, q, torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda())
    for r in range(nrows):
        expect = (48 * -2.0 + priv_tokens[r] * (r + 1) / 8) / ctx[r]
        G.assert_close(out[r], np.full((H, 128), expect), f"row {r}")


def test_device_checks_skip_bad_tables_and_lengths(pkv):
    N, H = 16, 32
    pool = G.device_pool(N, 1, H, seed=4)
    p = pkv.Pool(pool, N, num_layers=1)
    q = workloads.normal_fp16((2, H, 128), 1).cuda()
    out = torch.zeros_like(q)
    tables = torch.tensor([[3, N + 5], [1, 2]], dtype=torch.int32, device="cuda")   # row 0 names a block past the pool
    p.decode_attn(0, q, tables, torch.tensor([20, 20], dtype=torch.int32, device="cuda"), G.SCALE, out)
    st, flags = p.get_status()
    assert st == pkv.PKV_E_DEVICE and flags & pkv.PKV_DEV_BAD_BLOCK
    p.decode_attn(0, q, tables, torch.tensor([33, 0], dtype=torch.int32, device="cuda"), G.SCALE, out)
    st, flags = p.get_status()
    assert st == pkv.PKV_E_DEVICE and flags & pkv.PKV_DEV_BAD_CTX
    # a correct call afterwards still works
    good = torch.tensor([[3, 4], [1, 2]], dtype=torch.int32, device="cuda")
    _decode(pkv, p, 0, q, good, torch.tensor([20, 32], dtype=torch.int32, device="cuda"))


def test_host_refuses_bad_arguments(pkv):
    N = 8
    pool = G.device_pool(N, 2, 32, seed=5)
    p = pkv.Pool(pool, N, num_layers=2)
    q = torch.zeros(2, 32, 128, dtype=torch.float16, device="cuda")
    t = torch.zeros(2, 4, dtype=torch.int32, device="cuda")
    c = torch.ones(2, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError):
        p.decode_attn(2, q, t, c, G.SCALE, q)                       # layer out of range
    with pytest.raises(pkv.PkvError):
        p.decode_attn(0, q, torch.zeros(2, 200, dtype=torch.int32, device="cuda"), c, G.SCALE, q)  # no workspace
    with pytest.raises(pkv.PkvError):
        p.kv_append(0, q[:, :, 1:], q, torch.zeros(2, dtype=torch.int64, device="cuda"))           # misaligned k


def test_bounded_wait_times_out_and_returns(pkv):
    pool = G.device_pool(4, 1, 32, seed=6)
    p = pkv.Pool(pool, 4, num_layers=1)
    p.debug_wait_probe(2_000_000)             # 2 ms; nothing ever arrives on the barrier
    st, flags = p.get_status()
    assert st == pkv.PKV_E_TIMEOUT and flags & pkv.PKV_DEV_TIMEOUT
    assert p.get_status() == (pkv.PKV_OK, 0)


def test_step_matches_per_layer_calls(pkv):
    wl = workloads.random_step(21, num_seqs=7, max_ctx=900, num_blocks=500, num_layers=4)
    L, T, H = wl.num_layers, wl.num_tokens, wl.num_heads
    pool_a = G.device_pool(wl.num_blocks, L, H, seed=21)
    pool_b = pool_a.clone()
    pa = pkv.Pool(pool_a, wl.num_blocks, num_layers=L)
    pb = pkv.Pool(pool_b, wl.num_blocks, num_layers=L)
    tables_d, ctx_d, qs_d, slots_d, _ = G.step_metadata(wl)
    qkv = [G.new_token_inputs(wl, l) for l in range(L)]
    q = torch.stack([x[0] for x in qkv])
    k = torch.stack([x[1] for x in qkv])
    v = torch.stack([x[2] for x in qkv])
    out_a = torch.empty_like(q)
    for l in range(L):
        pa.kv_append(l, k[l], v[l], slots_d)
        out_a[l] = _decode(pkv, pa, l, q[l], tables_d, ctx_d)
    out_b = torch.empty_like(q)
    sd = pkv.make_step_desc(num_decode=T, num_prefill=0, num_tokens=T, max_q_len=0, max_blocks=wl.max_blocks,
                            first_layer=0, num_layers=L, scale=G.SCALE, block_tables=tables_d, ctx_lens=ctx_d,
                            q_start_loc=qs_d, slot_mapping=slots_d, q=q, k=k, v=v, out=out_b,
                            q_layer_stride=T * H * 128, k_layer_stride=T * H * 128, v_layer_stride=T * H * 128,
                            out_layer_stride=T * H * 128)
    ws = torch.empty(pb.step_workspace_bytes(sd), dtype=torch.uint8, device="cuda")
    pb.step(sd, ws)
    assert pb.get_status() == (pkv.PKV_OK, 0)
    assert torch.equal(out_a, out_b)
    assert torch.equal(pool_a, pool_b)
