"""GPU parity of the 8-bit KV cache against the oracle.

kv_append into an INT8 pool quantises each (token, head) row of K and V:
scale = max|x| / 127, code = round-half-even(x / scale) in IEEE single
precision; the stored codes and scales must equal the oracle's bit for bit
(untouched rows too). Decode and prefill attention read code * scale; their
outputs must satisfy |gpu - ref| <= 2e-3 + 1e-2 |ref| against the oracle's
double precision attention over the same pool.
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
    return t.detach().cpu().contiguous().numpy().reshape(-1).copy()


def _rows(shape, seed, special=False):
    """FP16 K/V rows: N(0,1), and with `special` some rows scaled to extremes, a zero row and ties."""
    x = workloads.normal_fp16(shape, seed).numpy().astype(np.float32)
    if special:
        T = shape[0]
        x[0] = 0.0                                   # zero row: scale 0, codes 0
        x[1 % T] *= 3e4 / max(1e-6, np.abs(x[1 % T]).max())   # near the FP16 maximum
        x[2 % T] *= 1e-6                             # subnormal FP16 values
        x[3 % T] = np.round(np.linspace(-127, 127, shape[-1]))[None, :] * 0.5   # exact codes and .5 cases
    return torch.from_numpy(x.astype(np.float16))


@pytest.mark.parametrize("layer,T", [(0, 1), (2, 37), (1, 300)])
def test_int8_kv_append_bit_exact_and_canaries_untouched(pkv, layer, T):
    N, L, H = 40, 3, 32
    pool = G.device_pool_i8(N, L, H, seed=1)
    host = _bytes(pool)
    p = pkv.Pool(pool, N, num_layers=L, num_heads=H, dtype="int8")
    rng = np.random.default_rng(T)
    slots = rng.choice(N * 16, T, replace=False).astype(np.int64)
    k = _rows((T, H, 128), 11 + T, special=True).cuda()
    v = _rows((T, H, 128), 12 + T).cuda()
    p.kv_append(layer, k, v, torch.from_numpy(slots).cuda())
    assert p.get_status() == (pkv.PKV_OK, 0)
    g = oracle.geom(N, L, H, dtype=oracle.INT8)
    assert oracle.kv_append(host, g, layer, G.to_bits(k), G.to_bits(v), slots) == -1
    assert np.array_equal(_bytes(pool), host)


def test_int8_kv_append_rejects_bad_slot(pkv):
    N, L, H = 8, 1, 4
    pool = G.device_pool_i8(N, L, H, seed=2)
    before = _bytes(pool)
    p = pkv.Pool(pool, N, num_layers=L, num_heads=H, dtype="int8")
    k = torch.ones(2, H, 128, dtype=torch.float16, device="cuda")
    p.kv_append(0, k, k, torch.tensor([N * 16, -5], dtype=torch.int64, device="cuda"))
    st, flags = p.get_status()
    assert st == pkv.PKV_E_DEVICE and flags & pkv.PKV_DEV_BAD_SLOT
    assert np.array_equal(_bytes(pool), before)


def run_i8(pkv, wl, partition=0, use_step=False, layers=None, garbage_tail=False, hq=None):
    """hq: query heads (default the pool's K/V heads); query head h reads K/V head h // (hq // heads)."""
    L, H, T, B = wl.num_layers, wl.num_heads, wl.num_tokens, wl.num_decode
    hq = hq or H
    assert B == wl.num_seqs
    layers = list(range(L)) if layers is None else layers
    pool = G.device_pool_i8(wl.num_blocks, L, H, seed=wl.seed)
    if garbage_tail:
        # rows past each row's context in its last block: codes -128 and NaN scales
        t5 = pool.view(wl.num_blocks, L, 2, H, 2112)
        for r in range(wl.num_seqs):
            c = int(wl.ctx_lens[r])
            if c % 16:
                b = int(wl.block_tables[r, c // 16])
                t5[b, :, :, :, (c % 16) * 128:2048] = 0x80
                sc = t5[b, :, :, :, 2048:].clone().view(torch.float32)
                sc[..., c % 16:] = float("nan")
                t5[b, :, :, :, 2048:] = sc.view(torch.uint8)
    host = _bytes(pool)
    p = pkv.Pool(pool, wl.num_blocks, num_layers=L, num_heads=H, partition_tokens=partition, dtype="int8",
                 num_q_heads=hq)
    tables_d, ctx_d, qs_d, slots_d, slots = G.step_metadata(wl)
    qkv = [G.new_token_inputs(wl, l) for l in range(L)]
    q = torch.stack([workloads.normal_fp16((T, hq, 128), workloads.value_seed(wl.seed, "q", l)) for l in range(L)])
    q = q.cuda().contiguous()
    k = torch.stack([x[1] for x in qkv]).contiguous()
    v = torch.stack([x[2] for x in qkv]).contiguous()
    out = torch.full_like(q, float("nan"))
    if use_step:
        sd = pkv.make_step_desc(num_decode=B, num_prefill=0, num_tokens=T, max_q_len=0, max_blocks=wl.max_blocks,
                                first_layer=0, num_layers=L, scale=G.SCALE, block_tables=tables_d, ctx_lens=ctx_d,
                                q_start_loc=qs_d, slot_mapping=slots_d, q=q, k=k, v=v, out=out,
                                q_layer_stride=T * hq * 128, k_layer_stride=T * H * 128, v_layer_stride=T * H * 128,
                                out_layer_stride=T * hq * 128)
        ws = torch.empty(max(p.step_workspace_bytes(sd), 256), dtype=torch.uint8, device="cuda")
        p.step(sd, ws)
    else:
        ws = torch.empty(max(p.decode_workspace_bytes(B, wl.max_blocks), 256), dtype=torch.uint8, device="cuda")
        for l in range(L):
            p.kv_append(l, k[l], v[l], slots_d)
            p.decode_attn(l, q[l], tables_d, ctx_d, G.SCALE, out[l], ws)
    st, flags = p.get_status()
    assert st == pkv.PKV_OK and flags == 0, (st, flags)
    g = oracle.geom(wl.num_blocks, L, H, dtype=oracle.INT8, num_q_heads=hq)
    for l in range(L):
        assert oracle.kv_append(host, g, l, G.to_bits(k[l]), G.to_bits(v[l]), slots) == -1
        if l in layers:
            ref, _ = oracle.decode_attn(host, g, l, G.to_bits(q[l]), wl.block_tables, wl.ctx_lens, G.SCALE)
            G.assert_close(out[l], ref, f"int8 decode layer {l}")
    if not garbage_tail:
        assert np.array_equal(_bytes(pool), host), "pool differs from the oracle's after append"
    return out


def _wl(seed, num_seqs=9, max_ctx=1500, num_layers=2, min_ctx=1, edges=True):
    nb = num_seqs * (-(-max_ctx // 16)) + 16
    wl = workloads.random_step(seed, num_seqs=num_seqs, max_ctx=max_ctx, num_blocks=nb, num_layers=num_layers,
                               min_ctx=min_ctx)
    if edges:
        wl.ctx_lens[0] = 1
        wl.ctx_lens[1] = 16
        wl.ctx_lens[2] = 17
    return wl


def test_int8_tiny_decode_config(pkv):
    run_i8(pkv, workloads.tiny_decode(0))


@pytest.mark.parametrize("seed", [1, 2])
@pytest.mark.parametrize("partition", [0, 64, 2048, 4096])
def test_int8_random_ragged_decode(pkv, seed, partition):
    run_i8(pkv, _wl(seed), partition)


def test_int8_fused_append_in_step_equals_separate(pkv):
    wl = _wl(5, max_ctx=2500)
    a = run_i8(pkv, wl, partition=256, use_step=True)
    b = run_i8(pkv, wl, partition=256, use_step=False)
    assert torch.equal(a, b)


def test_int8_long_rows_many_partitions(pkv):
    wl = _wl(7, num_seqs=3, max_ctx=4200, min_ctx=3000, num_layers=1, edges=False)
    run_i8(pkv, wl, partition=64)


def test_int8_ignores_garbage_past_the_context(pkv):
    run_i8(pkv, _wl(8), garbage_tail=True)
    run_i8(pkv, _wl(8), garbage_tail=True, use_step=True)


def test_int8_batch_invariance(pkv):
    wl = _wl(11, num_seqs=10, max_ctx=2600, num_layers=1)
    pool = G.device_pool_i8(wl.num_blocks, 1, 32, seed=11)
    p = pkv.Pool(pool, wl.num_blocks, num_layers=1, dtype="int8")
    tables_d, ctx_d, _, _, _ = G.step_metadata(wl)
    q, _, _ = G.new_token_inputs(wl, 0)
    ws = torch.empty(p.decode_workspace_bytes(wl.num_seqs, wl.max_blocks), dtype=torch.uint8, device="cuda")
    together = torch.empty_like(q)
    p.decode_attn(0, q, tables_d, ctx_d, G.SCALE, together, ws)
    for r in range(wl.num_seqs):
        alone = torch.empty_like(q[r:r + 1])
        p.decode_attn(0, q[r:r + 1].contiguous(), tables_d[r:r + 1].contiguous(), ctx_d[r:r + 1].contiguous(),
                      G.SCALE, alone, ws)
        assert torch.equal(alone[0], together[r])
    assert p.get_status() == (pkv.PKV_OK, 0)


def test_int8_close_to_fp16_decode(pkv):
    # quantisation error, not parity: the same appended N(0,1) values attended through an FP16 and an INT8 pool
    wl = _wl(12, num_seqs=6, max_ctx=1200, num_layers=1, edges=False)
    tables_d, ctx_d, _, slots_d, _ = G.step_metadata(wl)
    N, H = wl.num_blocks, 32
    allslots = torch.arange(N * 16, dtype=torch.int64, device="cuda")
    kk = workloads.normal_fp16((N * 16, H, 128), 21).cuda()
    vv = workloads.normal_fp16((N * 16, H, 128), 22).cuda()
    p16 = pkv.Pool(torch.empty(workloads.pool_shape(N, 1, H), dtype=torch.float16, device="cuda"), N, num_layers=1)
    p8 = pkv.Pool(torch.empty(pkv.Pool.bytes_needed(N, 1, H, "int8"), dtype=torch.uint8, device="cuda"), N,
                  num_layers=1, dtype="int8")
    q, _, _ = G.new_token_inputs(wl, 0)
    ws = torch.empty(p16.decode_workspace_bytes(wl.num_seqs, wl.max_blocks), dtype=torch.uint8, device="cuda")
    outs = []
    for p in (p16, p8):
        p.kv_append(0, kk, vv, allslots)
        o = torch.empty_like(q)
        p.decode_attn(0, q, tables_d, ctx_d, G.SCALE, o, ws)
        assert p.get_status() == (pkv.PKV_OK, 0)
        outs.append(o.double())
    err = (outs[0] - outs[1]).abs().max().item()
    assert 0 < err < 0.02, err


# (query heads, K/V heads): G = 4, MQA, G = 12 (fragment rows past 8), G = 32 (two slices), G = 3; and G = 2, 5,
# 7, 8: up to 8 query heads a CTA take the transposed form (query heads as the MMA's 8 columns), odd counts
# leaving a column pair half used
@pytest.mark.parametrize("hq,h", [(32, 8), (16, 1), (48, 4), (64, 2), (6, 2), (8, 4), (20, 4), (14, 2), (16, 2)])
@pytest.mark.parametrize("use_step", [False, True])
def test_int8_grouped_query_heads(pkv, hq, h, use_step):
    wl = _wl(hq + h, num_seqs=7, max_ctx=1300)
    wl.num_heads = h
    run_i8(pkv, wl, partition=128 if use_step else 0, use_step=use_step, hq=hq)


def _mixed_wl(ctx, qlen, seed=0, num_layers=1):
    """Explicit rows: q_len 1 rows are decode rows and come first, then prefill chunks."""
    ctx = np.asarray(ctx, np.int32)
    qlen = np.asarray(qlen, np.int32)
    nb = [-(-int(c) // 16) for c in ctx]
    N = sum(nb) + 8
    perm = np.random.default_rng(seed).permutation(N).astype(np.int32)
    tables = np.full((len(ctx), max(nb)), -1, np.int32)
    cur = 0
    for r, b in enumerate(nb):
        tables[r, :b] = perm[cur:cur + b]
        cur += b
    return workloads.Workload(f"i8mixed{seed}", num_layers, N, tables, ctx, qlen, seed)


def run_i8_prefill(pkv, wl, use_step, hq=None, garbage_tail=False):
    """Append (quantising) then attend: decode rows and prefill chunks over an 8-bit pool, against the
    oracle's double-precision attention over its own appended copy of the pool."""
    L, H, T, B = wl.num_layers, wl.num_heads, wl.num_tokens, wl.num_decode
    hq = hq or H
    pool = G.device_pool_i8(wl.num_blocks, L, H, seed=wl.seed)
    if garbage_tail:
        # positions past each row's context in its last block: codes -128 and NaN scales
        t5 = pool.view(wl.num_blocks, L, 2, H, 2112)
        for r in range(wl.num_seqs):
            c = int(wl.ctx_lens[r])
            if c % 16:
                b = int(wl.block_tables[r, c // 16])
                t5[b, :, :, :, (c % 16) * 128:2048] = 0x80
                sc = t5[b, :, :, :, 2048:].clone().view(torch.float32)
                sc[..., c % 16:] = float("nan")
                t5[b, :, :, :, 2048:] = sc.view(torch.uint8)
    host = _bytes(pool)
    p = pkv.Pool(pool, wl.num_blocks, num_layers=L, num_heads=H, dtype="int8", num_q_heads=hq)
    tables_d, ctx_d, qs_d, slots_d, slots = G.step_metadata(wl)
    q = torch.stack([workloads.normal_fp16((T, hq, 128), workloads.value_seed(wl.seed, "q", l)) for l in range(L)])
    q = q.cuda().contiguous()
    k = torch.stack([workloads.normal_fp16((T, H, 128), workloads.value_seed(wl.seed, "k", l)) for l in range(L)])
    v = torch.stack([workloads.normal_fp16((T, H, 128), workloads.value_seed(wl.seed, "v", l)) for l in range(L)])
    k, v = k.cuda().contiguous(), v.cuda().contiguous()
    out = torch.full_like(q, float("nan"))
    max_q = int(wl.q_lens[B:].max())
    if use_step:
        sd = pkv.make_step_desc(num_decode=B, num_prefill=wl.num_seqs - B, num_tokens=T, max_q_len=max_q,
                                max_blocks=wl.max_blocks, first_layer=0, num_layers=L, scale=G.SCALE,
                                block_tables=tables_d, ctx_lens=ctx_d, q_start_loc=qs_d, slot_mapping=slots_d,
                                q=q, k=k, v=v, out=out, q_layer_stride=T * hq * 128, k_layer_stride=T * H * 128,
                                v_layer_stride=T * H * 128, out_layer_stride=T * hq * 128)
        ws = torch.empty(max(p.step_workspace_bytes(sd), 256), dtype=torch.uint8, device="cuda")
        p.step(sd, ws)
    else:
        ws = torch.empty(max(p.decode_workspace_bytes(max(B, 1), wl.max_blocks), 256), dtype=torch.uint8,
                         device="cuda")
        for l in range(L):
            p.kv_append(l, k[l], v[l], slots_d)
            if B:
                p.decode_attn(l, q[l, :B], tables_d[:B], ctx_d[:B], G.SCALE, out[l, :B], ws)
            p.prefill_attn(l, q[l], qs_d[B:], tables_d[B:], ctx_d[B:], max_q, G.SCALE, out[l])
    st, flags = p.get_status()
    assert st == pkv.PKV_OK and flags == 0, (st, flags)
    g = oracle.geom(wl.num_blocks, L, H, dtype=oracle.INT8, num_q_heads=hq)
    qs = wl.q_start_loc()
    for l in range(L):
        assert oracle.kv_append(host, g, l, G.to_bits(k[l]), G.to_bits(v[l]), slots) == -1
        if B:
            ref, _ = oracle.decode_attn(host, g, l, G.to_bits(q[l, :B]), wl.block_tables[:B], wl.ctx_lens[:B],
                                        G.SCALE)
            G.assert_close(out[l, :B], ref, f"int8 decode rows layer {l}")
        ref, _ = oracle.prefill_attn(host, g, l, G.to_bits(q[l, qs[B]:]), qs[B:] - qs[B], wl.block_tables[B:],
                                     wl.ctx_lens[B:], G.SCALE)
        G.assert_close(out[l, qs[B]:], ref, f"int8 prefill layer {l}")
    if not garbage_tail:
        assert np.array_equal(_bytes(pool), host), "pool differs from the oracle's after append"
    return out


# (ctx, q_len) per row: decode rows first (q_len 1). Covers a fresh prompt shorter than one tile, chunks
# over a cached prefix with ragged last tiles and partial query tiles, several query tiles, one key block,
# chunks of two and three tokens.
I8_PREFILL_CASES = {
    "fresh_prompt": ([100], [100]),
    "chunk_over_prefix": ([700], [200]),
    "mixed": ([37, 300, 1290, 513, 16], [1, 1, 400, 129, 16]),
    "tiny_chunks": ([1, 2, 130], [1, 2, 3]),
    "long": ([2100, 1000], [512, 130]),
}


@pytest.mark.parametrize("case", sorted(I8_PREFILL_CASES))
@pytest.mark.parametrize("use_step", [False, True])
def test_int8_prefill(pkv, case, use_step):
    ctx, ql = I8_PREFILL_CASES[case]
    run_i8_prefill(pkv, _mixed_wl(ctx, ql, seed=len(case), num_layers=2), use_step)


@pytest.mark.parametrize("hq,h", [(32, 8), (8, 1)])
def test_int8_prefill_grouped_query_heads(pkv, hq, h):
    wl = _mixed_wl([33, 900, 300], [1, 260, 300], seed=3)
    wl.num_heads = h
    run_i8_prefill(pkv, wl, use_step=True, hq=hq)


def test_int8_prefill_ignores_garbage_past_the_context(pkv):
    run_i8_prefill(pkv, _mixed_wl([45, 610, 333], [1, 300, 333], seed=4), use_step=False, garbage_tail=True)


def test_int8_prefill_close_to_fp16(pkv):
    # quantisation error, not parity: the same N(0,1) K/V attended by one chunk through FP16 and INT8 pools
    N, H, ctx, ql = 80, 32, 1200, 300
    tables = torch.arange(N, dtype=torch.int32, device="cuda")[None, :ctx // 16 + 1].contiguous()
    ctx_d = torch.tensor([ctx], dtype=torch.int32, device="cuda")
    qs = torch.tensor([0, ql], dtype=torch.int32, device="cuda")
    allslots = torch.arange(N * 16, dtype=torch.int64, device="cuda")
    kk = workloads.normal_fp16((N * 16, H, 128), 31).cuda()
    vv = workloads.normal_fp16((N * 16, H, 128), 32).cuda()
    q = workloads.normal_fp16((ql, H, 128), 33).cuda()
    p16 = pkv.Pool(torch.empty(workloads.pool_shape(N, 1, H), dtype=torch.float16, device="cuda"), N, num_layers=1)
    p8 = pkv.Pool(torch.empty(pkv.Pool.bytes_needed(N, 1, H, "int8"), dtype=torch.uint8, device="cuda"), N,
                  num_layers=1, dtype="int8")
    outs = []
    for p in (p16, p8):
        p.kv_append(0, kk, vv, allslots)
        o = torch.empty_like(q)
        p.prefill_attn(0, q, qs, tables, ctx_d, ql, G.SCALE, o)
        assert p.get_status() == (pkv.PKV_OK, 0)
        outs.append(o.double())
    err = (outs[0] - outs[1]).abs().max().item()
    assert 0 < err < 0.02, err