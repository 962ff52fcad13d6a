"""Pins for the oracle: facts fixed by the pages or by mathematics, not by the oracle itself.

Every oracle function is checked here against something independent of its
own code: the pages' printed arithmetic (tests/golden/page_arithmetic.txt),
numpy's binary16 conversion, numpy's C-order indexing of the block layout,
closed forms of softmax attention (one-hot and uniform), invariance under a
permutation of physical blocks, torch's float64 attention on contiguous
inputs, and the identities between chunked and unchunked prefill and between
split and unsplit decode. tests/test_oracle_mutants.py plants mistakes in a
copy of the oracle and checks that this file catches each of them.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_arithmetic.txt")
SCALE = oracle.SCALE_FP32


def _golden_lines():
    out = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                lhs, rhs = line.split("=")
                out.append((lhs.split(), int(rhs)))
    return out


def _geom_bytes(L, H, D, eb, bs, nblocks=1):
    assert int(eb) == 2
    return oracle.geom(nblocks, int(L), int(H), int(D), int(bs))


def _eval_golden(args):
    kind = args[0]
    if kind == "bytes_per_token":
        return oracle.bytes_per_token(_geom_bytes(*args[1:6]))
    if kind == "bytes_per_block":
        return oracle.bytes_per_block(_geom_bytes(*args[1:6]))
    if kind in ("pool_blocks", "pool_tokens"):
        g = _geom_bytes(*args[1:6])
        budget = int(args[6])
        n = budget // oracle.bytes_per_block(g)
        # the next block would not fit
        assert oracle.pool_bytes(_geom_bytes(*args[1:6], nblocks=n + 1)) > budget
        assert oracle.pool_bytes(_geom_bytes(*args[1:6], nblocks=n)) <= budget
        return n if kind == "pool_blocks" else n * int(args[5])
    if kind == "request_bytes":
        return oracle.bytes_per_token(_geom_bytes(*args[1:6])) * int(args[6])
    if kind == "requests_fit":
        g = _geom_bytes(*args[1:6])
        n = int(args[6]) // oracle.bytes_per_block(g)
        return n // oracle.blocks_for_tokens(int(args[7]), int(args[5]))
    if kind == "batch_gb_rounded":
        g = _geom_bytes(*args[1:6])
        return round(oracle.bytes_per_token(g) * int(args[6]) * int(args[7]) / 1e9)
    if kind == "blocks_for":
        return oracle.blocks_for_tokens(int(args[2]), int(args[1]))
    if kind == "blocks_for_list":
        return sum(oracle.blocks_for_tokens(int(x), int(args[1])) for x in args[2].split(","))
    if kind == "slots_for_list":
        return sum(oracle.blocks_for_tokens(int(x), int(args[1])) * int(args[1]) for x in args[2].split(","))
    if kind == "unused_slots_list":
        xs = [int(x) for x in args[2].split(",")]
        return sum(oracle.blocks_for_tokens(x, int(args[1])) * int(args[1]) for x in xs) - sum(xs)
    if kind == "request_block_bytes":
        g = _geom_bytes(*args[1:6])
        return oracle.blocks_for_tokens(int(args[6]), int(args[5])) * int(args[5]) * oracle.bytes_per_token(g)
    raise KeyError(kind)


@pytest.mark.parametrize("args,expected", _golden_lines(), ids=lambda x: str(x)[:60])
def test_page_arithmetic(args, expected):
    assert _eval_golden(args) == expected


def test_scale_is_fp32_inverse_sqrt_128():
    assert np.float32(SCALE).view(np.uint32) == 0x3DB504F3


# ------------------------------------------------------------------ binary16

def test_half_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_half_encode_round_to_nearest_even():
    rng = np.random.default_rng(1)
    # every representable value, every midpoint between neighbours, and random doubles
    fin = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (fin[:-1] + fin[1:]) / 2
    rnd = np.concatenate([rng.standard_normal(100000) * s for s in (1e-6, 1e-3, 1.0, 100.0, 3e4)])
    x = np.concatenate([fin, mids, -mids, rnd, [65504.0, 65519.99, 65520.0, 1e6, -1e6, 0.0, -0.0]])
    ours = oracle.double_to_half(x)
    ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------------ helpers

def _pool(N, L, H, seed=0, D=128):
    t = workloads.normal_fp16(workloads.pool_shape(N, L, H, D), seed)
    return t.numpy().view(np.uint16).copy()


def _h(x):  # float array -> fp16 bits
    return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)


def _contig(pool6, layer, kv, head, table, n):
    """Contiguous K or V by numpy fancy indexing of [N, L, 2, H, 16, D]."""
    pos = np.arange(n)
    blk = np.asarray(table)[pos // 16]
    return pool6[blk, layer, kv, head, pos % 16, :].view(np.float16).astype(np.float64)


# ------------------------------------------------------------------ layout, append, gather

def test_kv_append_lands_at_numpy_layout():
    N, L, H = 12, 3, 4
    g = oracle.geom(N, L, H)
    pool = np.zeros(workloads.pool_shape(N, L, H), np.uint16)
    rng = np.random.default_rng(2)
    T = 9
    slots = rng.choice(N * 16, T, replace=False).astype(np.int64)
    k = rng.integers(0, 0x7c00, (T, H, 128)).astype(np.uint16)
    v = rng.integers(0, 0x7c00, (T, H, 128)).astype(np.uint16)
    assert oracle.kv_append(pool, g, 2, k, v, slots) == -1
    expect = np.zeros_like(pool)
    for i, s in enumerate(slots):
        expect[s // 16, 2, 0, :, s % 16, :] = k[i]
        expect[s // 16, 2, 1, :, s % 16, :] = v[i]
    assert np.array_equal(pool, expect)


@pytest.mark.parametrize("bad", [-1, 12 * 16])
def test_kv_append_rejects_out_of_range_slot(bad):
    N, L, H = 12, 1, 2
    g = oracle.geom(N, L, H)
    pool = np.zeros(workloads.pool_shape(N, L, H), np.uint16)
    k = np.ones((3, H, 128), np.uint16)
    assert oracle.kv_append(pool, g, 0, k, k, np.array([0, bad, 5], np.int64)) == 1
    assert not pool.any()


@pytest.mark.parametrize("n", [1, 15, 16, 17, 47, 64])
def test_append_then_gather_is_identity(n):
    N, L, H = 16, 2, 3
    g = oracle.geom(N, L, H)
    pool = np.zeros(workloads.pool_shape(N, L, H), np.uint16)
    rng = np.random.default_rng(n)
    table = rng.permutation(N)[: -(-n // 16)].astype(np.int32)
    rows = np.zeros((n, H, 128), np.uint16)
    for p in range(n):   # one token per step, as decode appends them
        k = _h(rng.standard_normal((1, H, 128)))
        slot = oracle.slots(table[None, :], np.zeros(1, np.int32), np.array([p]))
        assert oracle.kv_append(pool, g, 1, k, k, slot) == -1
        rows[p] = k[0]
    for h in range(H):
        for kv in (0, 1):
            got = oracle.gather(pool, g, 1, kv, h, table, n)
            assert np.array_equal(got, rows[:, h, :].view(np.float16).astype(np.float64))


def test_gather_reads_only_leading_rows_of_last_block():
    N, L, H = 4, 1, 1
    g = oracle.geom(N, L, H)
    pool6 = _pool(N, L, H)
    table = np.array([2, 0], np.int32)
    pool6[0, 0, :, 0, 1:, :] = 0x7e00          # NaN beyond the first row of the last block
    got = oracle.gather(pool6, g, 0, 0, 0, table, 17)
    assert not np.isnan(got).any()
    assert np.array_equal(got, _contig(pool6, 0, 0, 0, table, 17))


# ------------------------------------------------------------------ attention closed forms

def _decode_inputs(ctx, N=40, L=2, H=4, seed=3):
    rng = np.random.default_rng(seed)
    pool6 = _pool(N, L, H, seed)
    perm = rng.permutation(N).astype(np.int32)
    nb = [-(-c // 16) for c in ctx]
    tables = np.full((len(ctx), max(nb)), -1, np.int32)
    cur = 0
    for r, b in enumerate(nb):
        tables[r, :b] = perm[cur:cur + b]
        cur += b
    q = _h(rng.standard_normal((len(ctx), H, 128)))
    return pool6, oracle.geom(N, L, H), tables, np.array(ctx, np.int32), q


@pytest.mark.parametrize("j", [0, 15, 16, 31, 36])
def test_one_hot_softmax_returns_that_value_row(j):
    ctx = [37]
    pool6, g, tables, ctx, q = _decode_inputs(ctx)
    layer, H = 1, g.num_heads
    pos = np.arange(37)
    blk, off = tables[0][pos // 16], pos % 16
    pool6[blk, layer, 0] = 0
    # logits: q.k_j * scale ~ 128 * |q|^2 * scale >> 745, every other logit is 0
    pool6[blk[j], layer, 0, :, off[j], :] = _h(128.0 * q[0].view(np.float16).astype(np.float64))
    o64, o16 = oracle.decode_attn(pool6, g, layer, q, tables, ctx, SCALE)
    v_j = pool6[blk[j], layer, 1, :, off[j], :]
    assert np.array_equal(o64[0], v_j.view(np.float16).astype(np.float64))
    assert np.array_equal(o16[0], v_j)


def test_uniform_softmax_is_mean_of_values():
    pool6, g, tables, ctx, q = _decode_inputs([1, 16, 29, 100])
    pool6[:, :, 0] = 0
    o64, _ = oracle.decode_attn(pool6, g, 0, q, tables, ctx, SCALE)
    for r, n in enumerate(ctx):
        for h in range(g.num_heads):
            mean = _contig(pool6, 0, 1, h, tables[r], n).mean(axis=0)
            assert np.allclose(o64[r, h], mean, rtol=0, atol=1e-13)


def test_marker_rows_read_only_their_own_blocks():
    # 3 rows share 2 full prefix blocks; private values carry a per-row marker.
    N, L, H = 16, 1, 2
    g = oracle.geom(N, L, H)
    pool6 = np.zeros(workloads.pool_shape(N, L, H), np.uint16)
    shared = [5, 9]
    private = {0: [1], 1: [2, 3], 2: [4]}
    priv_tokens = [3, 20, 16]
    markers = [0.25, 0.5, -1.0]
    pool6[shared, :, 1] = _h(2.0)
    for r, blks in private.items():
        pool6[blks, :, 1] = _h(markers[r])
    for b in range(N):
        if b not in shared and all(b not in v for v in private.values()):
            pool6[b, :, 1] = _h(1000.0)       # foreign blocks: any read shows up
    tables = np.full((3, 4), -1, np.int32)
    for r in range(3):
        row = shared + private[r]
        tables[r, :len(row)] = row
    ctx = np.array([32 + t for t in priv_tokens], np.int32)
    q = _h(np.random.default_rng(0).standard_normal((3, H, 128)))
    o64, _ = oracle.decode_attn(pool6, g, 0, q, tables, ctx, SCALE)
    for r in range(3):
        expect = (32 * 2.0 + priv_tokens[r] * markers[r]) / ctx[r]
        assert np.allclose(o64[r], expect, rtol=0, atol=1e-12)


def test_physical_block_permutation_leaves_output_unchanged():
    pool6, g, tables, ctx, q = _decode_inputs([5, 33, 64, 90], N=40)
    o_ref, o16_ref = oracle.decode_attn(pool6, g, 1, q, tables, ctx, SCALE)
    rng = np.random.default_rng(7)
    perm = rng.permutation(g.num_blocks)          # block b moves to perm[b]
    moved = np.empty_like(pool6)
    moved[perm] = pool6
    t2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    o2, o16 = oracle.decode_attn(moved, g, 1, q, t2, ctx, SCALE)
    assert np.array_equal(o_ref, o2) and np.array_equal(o16_ref, o16)


def test_decode_matches_torch_float64_attention():
    pool6, g, tables, ctx, q = _decode_inputs([1, 2, 17, 50, 100, 255], N=40)
    o64, o16 = oracle.decode_attn(pool6, g, 1, q, tables, ctx, SCALE)
    for r, n in enumerate(ctx):
        for h in range(g.num_heads):
            K = torch.from_numpy(_contig(pool6, 1, 0, h, tables[r], n))
            V = torch.from_numpy(_contig(pool6, 1, 1, h, tables[r], n))
            qq = torch.from_numpy(q[r, h].view(np.float16).astype(np.float64))
            ref = torch.nn.functional.scaled_dot_product_attention(qq[None, None], K[None], V[None], scale=SCALE)[0, 0]
            assert np.allclose(o64[r, h], ref.numpy(), rtol=1e-12, atol=1e-13)
    assert np.array_equal(o16, oracle.double_to_half(o64))


# ------------------------------------------------------------------ grouped-query heads
# "Inference Infrastructure" (seeitflow), KV cache arithmetic: GQA shares one K/V head among a group of
# query heads, MQA one K/V head among all. A float64 library attention with the K/V heads repeated
# (query head h sees K/V head h // group) pins the oracle's grouped path.

def _gqa_case(ctx, hkv, hq, N=40, L=2, seed=11):
    pool6, _, tables, ctx, _ = _decode_inputs(ctx, N=N, L=L, H=hkv, seed=seed)
    q = _h(np.random.default_rng(seed + 1).standard_normal((len(ctx), hq, 128)))
    return pool6, oracle.geom(N, L, hkv, num_q_heads=hq), tables, ctx, q


@pytest.mark.parametrize("hkv,hq", [(2, 8), (1, 6), (3, 3)])
def test_gqa_decode_matches_torch_with_repeated_kv_heads(hkv, hq):
    pool6, g, tables, ctx, q = _gqa_case([1, 17, 50, 130], hkv, hq)
    o64, o16 = oracle.decode_attn(pool6, g, 1, q, tables, ctx, SCALE)
    assert o64.shape == (4, hq, 128)
    grp = hq // hkv
    for r, n in enumerate(ctx):
        K = torch.from_numpy(np.stack([_contig(pool6, 1, 0, k, tables[r], n) for k in range(hkv)]))
        V = torch.from_numpy(np.stack([_contig(pool6, 1, 1, k, tables[r], n) for k in range(hkv)]))
        Q = torch.from_numpy(q[r].view(np.float16).astype(np.float64))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K.repeat_interleave(grp, 0),
                                                               V.repeat_interleave(grp, 0), scale=SCALE)[:, 0]
        assert np.allclose(o64[r], ref.numpy(), rtol=1e-12, atol=1e-13)
    assert np.array_equal(o16, oracle.double_to_half(o64))


def test_gqa_equals_mha_with_each_kv_head_repeated():
    # an MHA pool whose query-head groups hold identical K/V heads gives the grouped result exactly
    hkv, hq = 2, 6
    pool6, g, tables, ctx, q = _gqa_case([33, 70], hkv, hq, N=20, L=1, seed=13)
    mha = np.ascontiguousarray(np.repeat(pool6, hq // hkv, axis=3))
    gm = oracle.geom(20, 1, hq)
    a64, a16 = oracle.decode_attn(pool6, g, 0, q, tables, ctx, SCALE)
    b64, b16 = oracle.decode_attn(mha, gm, 0, q, tables, ctx, SCALE)
    assert np.array_equal(a64, b64) and np.array_equal(a16, b16)
    qs = np.array([0, 33, 33 + 70], np.int32)
    qp = _h(np.random.default_rng(14).standard_normal((103, hq, 128)))
    c64, c16 = oracle.prefill_attn(pool6, g, 0, qp, qs, tables, ctx, SCALE)
    d64, d16 = oracle.prefill_attn(mha, gm, 0, qp, qs, tables, ctx, SCALE)
    assert np.array_equal(c64, d64) and np.array_equal(c16, d16)
    s64 = oracle.decode_attn_split(pool6, g, 0, q, tables, ctx, SCALE, 32)
    assert np.allclose(s64, a64, rtol=1e-12, atol=1e-14)


def test_gqa_prefill_matches_torch_causal_attention():
    n, hkv, hq = 70, 2, 8
    rng = np.random.default_rng(15)
    pool6 = _pool(12, 1, hkv, 15)
    table = rng.permutation(12)[: -(-n // 16)].astype(np.int32)
    q = _h(rng.standard_normal((n, hq, 128)))
    g = oracle.geom(12, 1, hkv, num_q_heads=hq)
    o64, _ = oracle.prefill_attn(pool6, g, 0, q, [0, n], table[None], [n], SCALE)
    mask = torch.ones(n, n, dtype=torch.bool).tril()
    for h in range(hq):
        K = torch.from_numpy(_contig(pool6, 0, 0, h // (hq // hkv), table, n))
        V = torch.from_numpy(_contig(pool6, 0, 1, h // (hq // hkv), table, n))
        Q = torch.from_numpy(q[:, h].view(np.float16).astype(np.float64))
        ref = torch.nn.functional.scaled_dot_product_attention(Q[None], K[None], V[None], attn_mask=mask[None],
                                                               scale=SCALE)[0]
        assert np.allclose(o64[:, h], ref.numpy(), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ prefill

def _prompt_case(n=70, N=12, L=1, H=3, seed=5):
    rng = np.random.default_rng(seed)
    pool6 = _pool(N, L, H, seed)
    table = rng.permutation(N)[: -(-n // 16)].astype(np.int32)
    q = _h(rng.standard_normal((n, H, 128)))
    return pool6, oracle.geom(N, L, H), table, q


def test_prefill_matches_torch_causal_attention():
    n = 70
    pool6, g, table, q = _prompt_case(n)
    o64, _ = oracle.prefill_attn(pool6, g, 0, q, [0, n], table[None], [n], SCALE)
    mask = torch.ones(n, n, dtype=torch.bool).tril()
    for h in range(g.num_heads):
        K = torch.from_numpy(_contig(pool6, 0, 0, h, table, n))
        V = torch.from_numpy(_contig(pool6, 0, 1, h, table, n))
        Q = torch.from_numpy(q[:, h].view(np.float16).astype(np.float64))
        ref = torch.nn.functional.scaled_dot_product_attention(Q[None], K[None], V[None], attn_mask=mask[None],
                                                               scale=SCALE)[0]
        assert np.allclose(o64[:, h], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_chunked_prefill_rows_equal_unchunked_rows():
    n, c = 70, 32
    pool6, g, table, q = _prompt_case(n)
    full64, full16 = oracle.prefill_attn(pool6, g, 0, q, [0, n], table[None], [n], SCALE)
    for s in range(0, n, c):
        e = min(s + c, n)
        o64, o16 = oracle.prefill_attn(pool6, g, 0, q[s:e], [0, e - s], table[None], [e], SCALE)
        assert np.array_equal(o64, full64[s:e]) and np.array_equal(o16, full16[s:e])


def test_decode_row_equals_last_prefill_row():
    n = 45
    pool6, g, table, q = _prompt_case(n)
    full64, _ = oracle.prefill_attn(pool6, g, 0, q, [0, n], table[None], [n], SCALE)
    d64, _ = oracle.decode_attn(pool6, g, 0, q[n - 1:n], table[None], [n], SCALE)
    assert np.array_equal(d64[0], full64[n - 1])


def test_prefill_several_sequences_in_one_call():
    pool6, g, tables, ctx, q_dec = _decode_inputs([20, 40, 35], N=40, L=1)
    qlens = [1, 7, 35]
    qs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = _h(np.random.default_rng(11).standard_normal((qs[-1], g.num_heads, 128)))
    o64, _ = oracle.prefill_attn(pool6, g, 0, q, qs, tables, ctx, SCALE)
    for s in range(3):
        for i in range(qlens[s]):
            pos = ctx[s] - qlens[s] + i
            d64, _ = oracle.decode_attn(pool6, g, 0, q[qs[s] + i:qs[s] + i + 1], tables[s:s + 1],
                                        np.array([pos + 1], np.int32), SCALE)
            assert np.array_equal(o64[qs[s] + i], d64[0])


# ------------------------------------------------------------------ split merge

@pytest.mark.parametrize("part", [16, 48, 100, 512, 4096])
def test_split_merge_equals_unsplit(part):
    pool6, g, tables, ctx, q = _decode_inputs([1, 16, 17, 250, 600], N=64)
    ref, _ = oracle.decode_attn(pool6, g, 0, q, tables, ctx, SCALE)
    got = oracle.decode_attn_split(pool6, g, 0, q, tables, ctx, SCALE, part)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_merge_of_two_halves_by_hand():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((30, 128))
    V = rng.standard_normal((30, 128))
    q = rng.standard_normal(128)
    m1, l1, o1 = oracle.partial(q, K, V, 0, 13, 0.1)
    m2, l2, o2 = oracle.partial(q, K, V, 13, 30, 0.1)
    got = oracle.merge([m1, m2], [l1, l2], np.stack([o1, o2]))
    s = 0.1 * K @ q
    p = np.exp(s - s.max())
    assert np.allclose(got, (p / p.sum()) @ V, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ 8-bit cache
# Reading (the pages fix no scale rule): INT8 codes, one float32 scale per (token, head) row of K or V,
# scale = max|x| / 127, code = round-half-even(x / scale); the stored value is code * scale.

def test_int8_codes_halve_the_pages_cache_figure():
    # "Inference Infrastructure" (seeitflow), KV cache arithmetic: 8 bits per element halve the cache, the
    # 512 MiB of a 4,096-token sequence (32 layers, 8 K/V heads, 128 dims) becoming 256 MiB. The scales
    # (4 B per row of 128 codes) are metadata on top ("The inference engine", quantisation costs).
    g16 = oracle.geom(1, 32, 8)
    g8 = oracle.geom(1, 32, 8, dtype=oracle.INT8)
    tile = oracle.i8_tile_bytes(g8)
    assert tile == 16 * 128 + 16 * 4
    code_bytes_per_token = 2 * 32 * 8 * (tile - 16 * 4) // 16
    assert code_bytes_per_token * 2 == oracle.bytes_per_token(g16) == 131072
    assert code_bytes_per_token * 4096 == 256 * 2**20
    assert oracle.bytes_per_token(g8) - code_bytes_per_token == 2 * 32 * 8 * 4
    # the 32-head model's 60 GB pool: 4,325,376 B per block, 13,871 blocks (7,152 at FP16)
    m8 = oracle.geom(1, 32, 32, dtype=oracle.INT8)
    assert oracle.bytes_per_block(m8) == 32 * 2 * 32 * tile == 4325376
    assert 60_000_000_000 // oracle.bytes_per_block(m8) == 13871


def _exact_rows(rng, n_rows, D=128, kmin=0, kmax=8):
    """Rows x = c * 2^-k with integer |c| <= 127 and max |c| = 127: exactly representable in FP16 and
    exactly recoverable from an INT8 code and a power-of-two scale."""
    c = rng.integers(-127, 128, (n_rows, D))
    c[np.arange(n_rows), rng.integers(0, D, n_rows)] = rng.choice([-127, 127], n_rows)
    k = rng.integers(kmin, kmax + 1, n_rows)
    s = np.ldexp(1.0, -k)
    x = (c * s[:, None]).astype(np.float16)
    assert np.array_equal(x.astype(np.float64), c * s[:, None])
    return x, c.astype(np.int8), s.astype(np.float32)


def test_int8_quantise_exactly_representable_rows():
    rng = np.random.default_rng(0)
    x, c, s = _exact_rows(rng, 200)
    for i in range(200):
        codes, scale = oracle.i8_quantize_row(x[i].view(np.uint16))
        assert scale == s[i]
        assert np.array_equal(codes, c[i])
        assert all(oracle.i8_dequant(int(codes[d]), scale) == float(x[i, d]) for d in range(0, 128, 17))


@pytest.mark.parametrize("mag", [1e-3, 1.0, 100.0])
def test_int8_quantise_error_bound_and_nearest_code(mag):
    rng = np.random.default_rng(int(mag * 1000) + 1)
    for _ in range(100):
        x = (rng.standard_normal(128) * mag).astype(np.float16)
        xd = x.astype(np.float64)
        codes, scale = oracle.i8_quantize_row(x.view(np.uint16))
        amax = np.abs(xd).max()
        assert abs(float(scale) - amax / 127) <= amax / 127 * 2.0**-23
        assert codes.min() >= -127 and codes.max() <= 127
        j = int(np.argmax(np.abs(xd)))
        assert int(codes[j]) == (127 if xd[j] > 0 else -127)
        # the nearest integer to x / scale (float64), away from exact midpoints
        r = xd / np.float64(scale)
        clear = np.abs(np.abs(r - np.floor(r)) - 0.5) > 1e-5
        assert np.array_equal(codes[clear].astype(np.int64), np.rint(r[clear]).astype(np.int64))
        back = np.array([oracle.i8_dequant(int(cc), scale) for cc in codes])
        assert np.all(np.abs(back - xd) <= float(scale) * (0.5 + 1e-5))


def test_int8_quantise_zero_row():
    codes, scale = oracle.i8_quantize_row(np.zeros(128, np.uint16))
    assert scale == 0 and not codes.any()


def _i8_case(rng, N=24, L=2, H=3, T=40):
    x_k, c_k, s_k = _exact_rows(rng, T * H)
    x_v, c_v, s_v = _exact_rows(rng, T * H)
    slots = rng.choice(N * 16, T, replace=False).astype(np.int64)
    return (x_k.reshape(T, H, 128), c_k.reshape(T, H, 128), s_k.reshape(T, H),
            x_v.reshape(T, H, 128), c_v.reshape(T, H, 128), s_v.reshape(T, H), slots)


def test_int8_append_places_codes_and_scales():
    # byte placement checked with numpy's own C-order view of [block, layer, K/V, head, tile bytes]
    rng = np.random.default_rng(3)
    N, L, H, T = 24, 2, 3, 40
    xk, ck, sk, xv, cv, sv, slots = _i8_case(rng, N, L, H, T)
    g = oracle.geom(N, L, H, dtype=oracle.INT8)
    pool = oracle.empty_pool(g)
    pool[:] = 0xA5
    layer = 1
    assert oracle.kv_append(pool, g, layer, xk.view(np.uint16), xv.view(np.uint16), slots) == -1
    tiles = pool.reshape(N, L, 2, H, 2112)
    touched = np.zeros((N, L, 2, H, 16), bool)
    for i, slot in enumerate(slots):
        b, t = divmod(int(slot), 16)
        for h in range(H):
            for kv, (c, s) in enumerate(((ck, sk), (cv, sv))):
                tile = tiles[b, layer, kv, h]
                assert np.array_equal(tile[t * 128:(t + 1) * 128].view(np.int8), c[i, h])
                assert tile[2048 + 4 * t:2048 + 4 * t + 4].view(np.float32)[0] == s[i, h]
                touched[b, layer, kv, h, t] = True
    # every other code row and scale is untouched
    for b in range(N):
        for l in range(L):
            for kv in range(2):
                for h in range(H):
                    for t in range(16):
                        if not touched[b, l, kv, h, t]:
                            assert (tiles[b, l, kv, h, t * 128:(t + 1) * 128] == 0xA5).all()
                            assert (tiles[b, l, kv, h, 2048 + 4 * t:2052 + 4 * t] == 0xA5).all()


def test_int8_attention_equals_fp16_attention_on_exact_values():
    # appended values that INT8 stores exactly: decode, split decode and prefill over the INT8 pool equal
    # the same computations over an FP16 pool holding the same values (pins INT8 gather and indexing
    # against the FP16 path, which the tests above pin)
    rng = np.random.default_rng(4)
    N, L, H, T = 24, 2, 3, 40
    xk, ck, sk, xv, cv, sv, _ = _i8_case(rng, N, L, H, T)
    perm = rng.permutation(N).astype(np.int32)
    ctx = np.array([40], np.int32)
    table = perm[None, :3]
    slots = oracle.slots(table, np.zeros(T, np.int32), np.arange(T))
    g16 = oracle.geom(N, L, H)
    g8 = oracle.geom(N, L, H, dtype=oracle.INT8)
    p16, p8 = oracle.empty_pool(g16), oracle.empty_pool(g8)
    for l in range(L):
        oracle.kv_append(p16, g16, l, xk.view(np.uint16), xv.view(np.uint16), slots)
        oracle.kv_append(p8, g8, l, xk.view(np.uint16), xv.view(np.uint16), slots)
    q = workloads.normal_fp16((T, H, 128), 9).numpy().view(np.uint16)
    for l in range(L):
        a16, _ = oracle.decode_attn(p16, g16, l, q[-1:], table, ctx, SCALE)
        a8, _ = oracle.decode_attn(p8, g8, l, q[-1:], table, ctx, SCALE)
        assert np.array_equal(a16, a8)
        s16 = oracle.decode_attn_split(p16, g16, l, q[-1:], table, ctx, SCALE, 16)
        s8 = oracle.decode_attn_split(p8, g8, l, q[-1:], table, ctx, SCALE, 16)
        assert np.array_equal(s16, s8)
        qs = np.array([0, T], np.int32)
        f16, _ = oracle.prefill_attn(p16, g16, l, q, qs, table, ctx, SCALE)
        f8, _ = oracle.prefill_attn(p8, g8, l, q, qs, table, ctx, SCALE)
        assert np.array_equal(f16, f8)


def test_int8_attention_close_to_fp16_attention_on_gaussian_values():
    # not a parity bound: the quantisation error of N(0,1) rows stays small against the FP16 result
    rng = np.random.default_rng(5)
    N, L, H, T = 40, 1, 4, 300
    k = workloads.normal_fp16((T, H, 128), 1).numpy().view(np.uint16)
    v = workloads.normal_fp16((T, H, 128), 2).numpy().view(np.uint16)
    q = workloads.normal_fp16((1, H, 128), 3).numpy().view(np.uint16)
    table = rng.permutation(N).astype(np.int32)[None, :19]
    slots = oracle.slots(table, np.zeros(T, np.int32), np.arange(T))
    g16, g8 = oracle.geom(N, L, H), oracle.geom(N, L, H, dtype=oracle.INT8)
    p16, p8 = oracle.empty_pool(g16), oracle.empty_pool(g8)
    oracle.kv_append(p16, g16, 0, k, v, slots)
    oracle.kv_append(p8, g8, 0, k, v, slots)
    a16, _ = oracle.decode_attn(p16, g16, 0, q, table, np.array([T], np.int32), SCALE)
    a8, _ = oracle.decode_attn(p8, g8, 0, q, table, np.array([T], np.int32), SCALE)
    assert np.abs(a16 - a8).max() < 0.02 and not np.array_equal(a16, a8)


# ------------------------------------------------------------------ block copy, swap, prefix hashes

def test_fnv1a64_published_vectors():
    # the FNV-1a 64-bit test values published with the algorithm (offset basis, "a", "foobar")
    assert oracle.fnv1a64(b"") == 0xCBF29CE484222325
    assert oracle.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert oracle.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_block_hash_chain_depends_on_the_whole_prefix():
    # "Serving LLMs" (sreshtalluri), "Prefix caching": a block's hash matches only if every earlier token
    # matches too; only full blocks are hashed.
    rng = np.random.default_rng(0)
    t = rng.integers(0, 50000, 16 * 9 + 7).astype(np.int32)
    h = oracle.block_hashes(t)
    assert h.shape == (9,)
    assert np.array_equal(oracle.block_hashes(t[:16 * 9]), h)          # the partial tail is not hashed
    assert np.array_equal(oracle.block_hashes(t[:16 * 4]), h[:4])      # a prefix's hashes are a prefix
    for j in [0, 15, 16, 70, 143]:
        u = t.copy()
        u[j] += 1
        hu = oracle.block_hashes(u)
        b = j // 16
        assert np.array_equal(hu[:b], h[:b]) and (hu[b:] != h[b:]).all()
    # block i's hash is FNV-1a over (previous hash, the block's 16 token ids), little-endian, from 0
    prev = 0
    for i in range(3):
        data = int(prev).to_bytes(8, "little") + t[16 * i:16 * i + 16].astype("<u4").tobytes()
        assert oracle.fnv1a64(data) == int(h[i])
        prev = int(h[i])


def test_copy_blocks_and_swap_are_whole_block_byte_copies():
    rng = np.random.default_rng(2)
    for dtype in (oracle.FP16, oracle.INT8):
        g = oracle.geom(12, 2, 3, dtype=dtype)
        pool = oracle.empty_pool(g)
        pool.view(np.uint8)[:] = rng.integers(0, 256, pool.nbytes, dtype=np.uint8)
        bb = oracle.bytes_per_block(g)
        view = pool.view(np.uint8).reshape(12, bb)
        expect = view.copy()
        pairs = np.array([[3, 7], [7, 1], [0, 11], [5, 5]], np.int32)    # in order: 7 <- 3, then 1 <- (new) 7
        for s_, d_ in pairs:
            expect[d_] = expect[s_]
        assert oracle.copy_blocks(pool, g, pairs) == -1
        assert np.array_equal(view, expect)
        before = view.copy()
        assert oracle.copy_blocks(pool, g, np.array([[1, 2], [3, 12]], np.int32)) == 1    # nothing copied
        assert np.array_equal(view, before)
        blocks = np.array([9, 0, 4, 4], np.int32)
        host = oracle.swap_out(pool, g, blocks)
        assert np.array_equal(host.reshape(4, bb), view[blocks])
        dst = np.array([2, 10, 6, 8], np.int32)
        assert oracle.swap_in(pool, g, dst, host) == -1
        assert np.array_equal(view[dst], before[blocks])
        with pytest.raises(IndexError):
            oracle.swap_out(pool, g, np.array([1, -1], np.int32))
