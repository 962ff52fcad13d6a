"""GPU parity of grouped-query and multi-query attention against the oracle.

The pool stores H K/V heads; the query has Hq = G x H heads and query head h
reads K/V head h // G ("Inference Infrastructure" (seeitflow), the KV cache
arithmetic: 8 K/V heads; one K/V head is multi-query attention). Each case
appends the step's new K/V, then attends through libpkv's C ABI; the oracle
applies its own kv_append to a host copy of the pool and computes attention in
double precision. Outputs must satisfy |gpu - ref| <= 2e-3 + 1e-2 |ref|, the
pool must match the oracle's bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _gpu as G
from tests.test_gpu_prefill import _wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return G.lib()


def _inputs(wl, layer, hq):
    T, H = wl.num_tokens, wl.num_heads
    q = workloads.normal_fp16((T, hq, 128), workloads.value_seed(wl.seed, "q", layer)).cuda()
    k = workloads.normal_fp16((T, H, 128), workloads.value_seed(wl.seed, "k", layer)).cuda()
    v = workloads.normal_fp16((T, H, 128), workloads.value_seed(wl.seed, "v", layer)).cuda()
    return q, k, v


def run_gqa(pkv, wl, hq, partition=0, use_step=True, nan_tail=False, layers=None):
    """Returns the attention output [L, T, hq, 128] after checking it (and the pool) against the oracle."""
    L, H, T, B = wl.num_layers, wl.num_heads, wl.num_tokens, wl.num_decode
    layers = list(range(L)) if layers is None else layers
    pool_t = G.device_pool(wl.num_blocks, L, H, seed=wl.seed)
    if nan_tail:
        for r in range(wl.num_seqs):
            c = int(wl.ctx_lens[r])
            if c % 16:
                pool_t[int(wl.block_tables[r, c // 16]), :, :, :, c % 16:, :] = float("nan")
    host = G.to_bits(pool_t).reshape(pool_t.shape).copy()
    p = pkv.Pool(pool_t, wl.num_blocks, num_layers=L, num_heads=H, partition_tokens=partition, num_q_heads=hq)
    tables_d, ctx_d, qs_d, slots_d, slots = G.step_metadata(wl)
    qkv = [_inputs(wl, l, hq) for l in range(L)]
    q = torch.stack([x[0] for x in qkv]).contiguous()
    k = torch.stack([x[1] for x in qkv]).contiguous()
    v = torch.stack([x[2] for x in qkv]).contiguous()
    out = torch.full_like(q, float("nan"))
    max_q = int(wl.q_lens[B:].max()) if wl.num_seqs > B else 0
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
            if wl.num_seqs > B:
                p.prefill_attn(l, q[l], qs_d[B:], tables_d[B:], ctx_d[B:], max_q, G.SCALE, out[l])
    st, flags = p.get_status()
    assert st == pkv.PKV_OK and flags == 0, (st, flags)
    g = oracle.geom(wl.num_blocks, L, H, num_q_heads=hq)
    qs = wl.q_start_loc()
    for l in range(L):
        assert oracle.kv_append(host, g, l, G.to_bits(k[l]), G.to_bits(v[l]), slots) == -1
        if l not in layers:
            continue
        if B:
            ref, _ = oracle.decode_attn(host, g, l, G.to_bits(q[l, :B]), wl.block_tables[:B], wl.ctx_lens[:B],
                                        G.SCALE)
            G.assert_close(out[l, :B], ref, f"decode rows, layer {l}, Hq {hq}, H {H}")
        if wl.num_seqs > B:
            ref, _ = oracle.prefill_attn(host, g, l, G.to_bits(q[l]), qs[B:], wl.block_tables[B:],
                                         wl.ctx_lens[B:], G.SCALE)
            G.assert_close(out[l, B:], ref[B:], f"prefill rows, layer {l}, Hq {hq}, H {H}")
    if not nan_tail:
        assert np.array_equal(G.to_bits(pool_t).reshape(pool_t.shape), host), "pool differs after append"
    return out


def _decode_wl(seed, heads, num_seqs=7, max_ctx=1300, num_blocks=None, num_layers=2, min_ctx=1, edges=True):
    num_blocks = num_blocks or num_seqs * (-(-max_ctx // 16)) + 16
    wl = workloads.random_step(seed, num_seqs=num_seqs, max_ctx=max_ctx, num_blocks=num_blocks,
                               num_layers=num_layers, min_ctx=min_ctx)
    wl.num_heads = heads
    if edges:
        wl.ctx_lens[0] = 1      # only the new token
        wl.ctx_lens[1] = 16     # exactly one full block
        wl.ctx_lens[2] = 17     # one full block and one token
    return wl


# (query heads, K/V heads): G = 4 (the 8-K/V-head model), MQA with 32 and 8 query
# heads, G = 12 (fragment rows past 8), G = 32 (two query-head slices per K/V
# head), G = 3 and G = 5 (rows that fill no power of two), G = 2.
GROUPS = [(32, 8), (32, 1), (8, 1), (48, 4), (64, 2), (6, 2), (40, 8), (16, 8)]


@pytest.mark.parametrize("hq,h", GROUPS)
@pytest.mark.parametrize("partition", [0, 64, 4096])
def test_gqa_decode_separate_append(pkv, hq, h, partition):
    run_gqa(pkv, _decode_wl(hq + h, h), hq, partition=partition, use_step=False)


@pytest.mark.parametrize("hq,h", GROUPS)
def test_gqa_decode_fused_append_in_step(pkv, hq, h):
    run_gqa(pkv, _decode_wl(100 + hq + h, h), hq, partition=128, use_step=True)


def test_gqa_fused_append_equals_separate(pkv):
    wl = _decode_wl(5, 8, num_seqs=9, max_ctx=2500)
    a = run_gqa(pkv, wl, 32, use_step=True)
    b = run_gqa(pkv, wl, 32, use_step=False)
    assert torch.equal(a, b)


@pytest.mark.parametrize("partition,ctxs", [(0, [1024, 1025, 1041, 2047, 2049, 2300, 3073]),
                                            (64, [64, 65, 127, 129, 1000, 2300, 3073]),
                                            (4096, [2300, 4096, 4097, 6000, 8193])])
def test_gqa_equal_partition_boundaries(pkv, partition, ctxs):
    # Equal-length partitions at and next to the bounds, with the decode rows' append fused into the last one.
    top = max(ctxs) + 30
    wl = _decode_wl(17, 8, num_seqs=len(ctxs), max_ctx=top, min_ctx=top, num_layers=1, edges=False)
    wl.ctx_lens[:] = ctxs
    run_gqa(pkv, wl, 32, partition=partition, use_step=True)


def test_gqa_long_rows_many_partitions(pkv):
    wl = _decode_wl(7, 8, num_seqs=3, max_ctx=4200, min_ctx=3000, num_layers=1, edges=False)
    assert wl.ctx_lens.min() >= 3000
    run_gqa(pkv, wl, 32, partition=64, use_step=False)


def test_gqa_ignores_nan_past_the_context(pkv):
    wl = _wl([75, 301, 33, 130], [1, 1, 1, 130], seed=6)
    wl.num_heads = 8
    run_gqa(pkv, wl, 32, nan_tail=True, use_step=False)
    run_gqa(pkv, wl, 32, nan_tail=True, use_step=True)


@pytest.mark.parametrize("ctx,qlen", [(70, 70), (300, 45), (256, 256), (1000, 300)])
@pytest.mark.parametrize("hq,h", [(32, 8), (8, 1)])
def test_gqa_prefill_one_sequence(pkv, ctx, qlen, hq, h):
    wl = _wl([ctx], [qlen], seed=ctx)
    wl.num_heads = h
    run_gqa(pkv, wl, hq, use_step=False)


def test_gqa_prefill_512_row_chunk_over_long_prefix_every_row(pkv):
    # the schedule's chunk 6 (512 queries after a 3,072-key prefix) with 2 K/V heads serving 8 query heads:
    # a CTA's 128 rows are 32 tokens of 4 query heads; every row against the oracle
    wl = _wl([3584], [512], seed=23)
    wl.num_heads = 2
    run_gqa(pkv, wl, 8, use_step=False)


@pytest.mark.parametrize("seed", [1, 2])
def test_gqa_mixed_step(pkv, seed):
    rng = np.random.default_rng(seed)
    dec_ctx = rng.integers(20, 900, 9).tolist()
    wl = _wl(dec_ctx + [600, 130], [1] * 9 + [300, 130], num_layers=2, seed=seed)
    wl.num_heads = 8
    run_gqa(pkv, wl, 32, partition=256)


def test_gqa_batch_invariance(pkv):
    wl = _decode_wl(11, 8, num_seqs=10, max_ctx=2600, num_layers=1)
    pool = G.device_pool(wl.num_blocks, 1, 8, seed=11)
    p = pkv.Pool(pool, wl.num_blocks, num_layers=1, num_heads=8, num_q_heads=32)
    tables_d, ctx_d, _, _, _ = G.step_metadata(wl)
    q = workloads.normal_fp16((wl.num_seqs, 32, 128), 3).cuda()
    ws = torch.empty(p.decode_workspace_bytes(wl.num_seqs, wl.max_blocks), dtype=torch.uint8, device="cuda")
    together = torch.empty_like(q)
    p.decode_attn(0, q, tables_d, ctx_d, G.SCALE, together, ws)
    for r in range(wl.num_seqs):
        alone = torch.empty_like(q[r:r + 1])
        p.decode_attn(0, q[r:r + 1].contiguous(), tables_d[r:r + 1].contiguous(), ctx_d[r:r + 1].contiguous(),
                      G.SCALE, alone, ws)
        assert torch.equal(alone[0], together[r])
    assert p.get_status() == (pkv.PKV_OK, 0)


def test_gqa_equals_mha_pool_with_repeated_heads(pkv):
    # A GQA pool and an MHA pool whose K/V heads are the GQA heads each repeated G times give the
    # same attention up to rounding (the two run different kernels).
    wl = _decode_wl(13, 4, num_seqs=5, max_ctx=900, num_layers=1)
    pool = G.device_pool(wl.num_blocks, 1, 4, seed=13)
    pg = pkv.Pool(pool, wl.num_blocks, num_layers=1, num_heads=4, num_q_heads=16)
    big = pool.repeat_interleave(4, dim=3).contiguous()
    pm = pkv.Pool(big, wl.num_blocks, num_layers=1, num_heads=16)
    tables_d, ctx_d, _, _, _ = G.step_metadata(wl)
    q = workloads.normal_fp16((wl.num_seqs, 16, 128), 4).cuda()
    ws = torch.empty(pm.decode_workspace_bytes(wl.num_seqs, wl.max_blocks), dtype=torch.uint8, device="cuda")
    a, b = torch.empty_like(q), torch.empty_like(q)
    pg.decode_attn(0, q, tables_d, ctx_d, G.SCALE, a, ws)
    pm.decode_attn(0, q, tables_d, ctx_d, G.SCALE, b, ws)
    assert pg.get_status() == (pkv.PKV_OK, 0)
    G.assert_close(a, G.to_f64(b), "GQA vs MHA with repeated heads")


def test_gqa_device_checks(pkv):
    N = 16
    pool = G.device_pool(N, 1, 8, seed=4)
    p = pkv.Pool(pool, N, num_layers=1, num_heads=8, num_q_heads=32)
    q = workloads.normal_fp16((2, 32, 128), 1).cuda()
    out = torch.zeros_like(q)
    tables = torch.tensor([[3, N + 5], [1, 2]], dtype=torch.int32, device="cuda")
    p.decode_attn(0, q, tables, torch.tensor([20, 20], dtype=torch.int32, device="cuda"), G.SCALE, out)
    st, flags = p.get_status()
    assert st == pkv.PKV_E_DEVICE and flags & pkv.PKV_DEV_BAD_BLOCK
    p.decode_attn(0, q, tables, torch.tensor([33, 0], dtype=torch.int32, device="cuda"), G.SCALE, out)
    st, flags = p.get_status()
    assert st == pkv.PKV_E_DEVICE and flags & pkv.PKV_DEV_BAD_CTX
    good = torch.tensor([[3, 4], [1, 2]], dtype=torch.int32, device="cuda")
    p.decode_attn(0, q, good, torch.tensor([20, 32], dtype=torch.int32, device="cuda"), G.SCALE, out)
    assert p.get_status() == (pkv.PKV_OK, 0)
