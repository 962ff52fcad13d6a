"""GPU parity of chunked causal prefill (tcgen05/TMEM) and of the mixed step
(decode rows + prefill chunks in one pkv_step) against the oracle.

Each case appends the step's new K/V (the chunk's own keys included), then
attends. The oracle applies its own kv_append to a host copy of the pool and
computes causal softmax attention in double precision; outputs must satisfy
|gpu - ref| <= 2e-3 + 1e-2 |ref|, the pool must match bit for bit.
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


def _wl(ctx, qlen, num_blocks=None, num_layers=1, seed=0):
    """Workload with explicit rows: q_len 1 rows are decode rows (they must come first)."""
    ctx = np.asarray(ctx, np.int32)
    qlen = np.asarray(qlen, np.int32)
    nb = [-(-int(c) // 16) for c in ctx]
    N = num_blocks or max(16, sum(nb) + 8)
    perm = np.random.default_rng(seed).permutation(N).astype(np.int32)
    tables = np.full((len(ctx), max(nb)), -1, np.int32)
    cur = 0
    for r, b in enumerate(nb):
        tables[r, :b] = perm[cur:cur + b]
        cur += b
    return workloads.Workload(f"case{seed}", num_layers, N, tables, ctx, qlen, seed)


def run_step_case(pkv, wl, layers=None, nan_tail=False, use_step=True):
    layers = list(range(wl.num_layers)) if layers is None else layers
    L, H, T = wl.num_layers, wl.num_heads, wl.num_tokens
    B = wl.num_decode
    pool_t = G.device_pool(wl.num_blocks, L, H, seed=wl.seed)
    if nan_tail:
        # positions past each row's context in its last block hold NaN
        for r in range(wl.num_seqs):
            c = int(wl.ctx_lens[r])
            if c % 16:
                pool_t[int(wl.block_tables[r, c // 16]), :, :, :, c % 16:, :] = float("nan")
    host = G.to_bits(pool_t).reshape(pool_t.shape).copy()
    p = pkv.Pool(pool_t, wl.num_blocks, num_layers=L, num_heads=H)
    tables_d, ctx_d, qs_d, slots_d, slots = G.step_metadata(wl)
    qkv = [G.new_token_inputs(wl, l) for l in range(L)]
    q = torch.stack([x[0] for x in qkv]).contiguous()
    k = torch.stack([x[1] for x in qkv]).contiguous()
    v = torch.stack([x[2] for x in qkv]).contiguous()
    out = torch.full_like(q, float("nan"))
    max_q = int(wl.q_lens[B:].max()) if wl.num_seqs > B else 0
    if use_step:
        sd = pkv.make_step_desc(num_decode=B, num_prefill=wl.num_seqs - B, num_tokens=T, max_q_len=max_q,
                                max_blocks=wl.max_blocks, first_layer=0, num_layers=L, scale=G.SCALE,
                                block_tables=tables_d, ctx_lens=ctx_d, q_start_loc=qs_d, slot_mapping=slots_d,
                                q=q, k=k, v=v, out=out, q_layer_stride=T * H * 128, k_layer_stride=T * H * 128,
                                v_layer_stride=T * H * 128, out_layer_stride=T * H * 128)
        ws = torch.empty(max(p.step_workspace_bytes(sd), 256), dtype=torch.uint8, device="cuda")
        p.step(sd, ws)
    else:
        for l in range(L):
            p.kv_append(l, k[l], v[l], slots_d)
            p.prefill_attn(l, q[l], qs_d[B:], tables_d[B:], ctx_d[B:], max_q, G.SCALE, out[l])
    st, flags = p.get_status()
    assert st == pkv.PKV_OK and flags == 0, (st, flags)
    g = oracle.geom(wl.num_blocks, L, H)
    qs = wl.q_start_loc()
    errs = []
    for l in range(L):
        assert oracle.kv_append(host, g, l, G.to_bits(k[l]), G.to_bits(v[l]), slots) == -1
        if l not in layers:
            continue
        if B and use_step:
            ref, _ = oracle.decode_attn(host, g, l, G.to_bits(q[l, :B]), wl.block_tables[:B], wl.ctx_lens[:B],
                                        G.SCALE)
            errs.append(G.assert_close(out[l, :B], ref, f"decode rows, layer {l}"))
        if wl.num_seqs > B:
            ref, _ = oracle.prefill_attn(host, g, l, G.to_bits(q[l]), qs[B:], wl.block_tables[B:],
                                         wl.ctx_lens[B:], G.SCALE)
            errs.append(G.assert_close(out[l, B:], ref[B:], f"prefill rows, layer {l}"))
    if not nan_tail:
        assert np.array_equal(G.to_bits(pool_t).reshape(pool_t.shape), host)
    return errs


@pytest.mark.parametrize("ctx,qlen", [(70, 70), (16, 16), (2, 2), (64, 64), (300, 45), (129, 129), (200, 200),
                                      (256, 256), (1000, 300), (777, 512), (4000, 416)])
def test_prefill_one_sequence(pkv, ctx, qlen):
    run_step_case(pkv, _wl([ctx], [qlen], seed=ctx), use_step=False)


def test_prefill_512_row_chunk_over_long_prefix_every_row(pkv):
    # a chunk of 512 queries at positions 3,072..3,583 (the schedule's chunk 6) over its 3,072-key prefix:
    # every row of every head against the oracle (4 heads keep the oracle's double-precision work small)
    wl = _wl([3584], [512], seed=21)
    wl.num_heads = 4
    run_step_case(pkv, wl, use_step=False)


def test_prefill_two_long_chunks_and_a_short_one_every_row(pkv):
    # several sequences with long prefixes in one call, ragged chunk lengths (a partial last query tile)
    wl = _wl([3100, 2049, 700], [300, 513, 129], seed=22)
    wl.num_heads = 2
    run_step_case(pkv, wl, use_step=False)


def test_prefill_several_sequences_one_call(pkv):
    run_step_case(pkv, _wl([200, 37, 513, 140], [200, 5, 260, 2], seed=5), use_step=False)


def test_prefill_ignores_nan_past_the_context(pkv):
    run_step_case(pkv, _wl([75, 301], [40, 301], seed=6), nan_tail=True, use_step=False)


def test_prefill_last_row_agrees_with_decode(pkv):
    ctx = 333
    wl = _wl([ctx], [ctx], seed=7)
    pool_t = G.device_pool(wl.num_blocks, 1, 32, seed=7)
    p = pkv.Pool(pool_t, wl.num_blocks, num_layers=1)
    tables_d, ctx_d, qs_d, _, _ = G.step_metadata(wl)
    q = workloads.normal_fp16((ctx, 32, 128), 17).cuda()
    out = torch.empty_like(q)
    p.prefill_attn(0, q, qs_d, tables_d, ctx_d, ctx, G.SCALE, out)
    dec = torch.empty(1, 32, 128, dtype=torch.float16, device="cuda")
    ws = torch.empty(p.decode_workspace_bytes(1, tables_d.shape[1]), dtype=torch.uint8, device="cuda")
    p.decode_attn(0, q[ctx - 1:].contiguous(), tables_d, ctx_d, G.SCALE, dec, ws)
    assert p.get_status() == (pkv.PKV_OK, 0)
    G.assert_close(out[ctx - 1:], G.to_f64(dec), "last prefill row vs decode")


@pytest.mark.parametrize("seed", [1, 2])
def test_mixed_step_decode_rows_and_prefill_chunk(pkv, seed):
    rng = np.random.default_rng(seed)
    dec_ctx = rng.integers(20, 900, 9).tolist()
    ctx = dec_ctx + [600, 130]
    qlen = [1] * 9 + [300, 130]
    run_step_case(pkv, _wl(ctx, qlen, num_layers=2, seed=seed))


@pytest.mark.parametrize("seed", [11, 12, 13, 14])
def test_mixed_step_random_ragged_batches(pkv, seed):
    # random batches: 0-3 decode rows, then 1-4 prefill rows of random context (1..1,500) and chunk length
    # (2..min(context, 300)), so query tiles end anywhere and chunks start inside blocks; 8 heads
    rng = np.random.default_rng(seed)
    nd, npf = int(rng.integers(0, 4)), int(rng.integers(1, 5))
    ctx = rng.integers(1, 1500, nd).tolist()
    qlen = [1] * nd
    for _ in range(npf):
        c = int(rng.integers(2, 1501))
        ctx.append(c)
        qlen.append(int(rng.integers(2, min(c, 300) + 1)))
    wl = _wl(ctx, qlen, num_layers=2, seed=seed)
    wl.num_heads = 8
    run_step_case(pkv, wl)


def test_mixed_chunk_schedule_small(pkv):
    # the chunked-prefill schedule of a 700-token prompt in 256-token chunks next to 5 decode rows
    for chunk in range(3):
        wl = workloads.mixed_prefill(chunk, seed=3, num_layers=1, num_blocks=1200, prompt_len=700, decode_rows=5,
                                     chunk_size=256)
        run_step_case(pkv, wl)


def test_prefill_device_checks(pkv):
    wl = _wl([100], [100], seed=8)
    pool_t = G.device_pool(wl.num_blocks, 1, 32, seed=8)
    p = pkv.Pool(pool_t, wl.num_blocks, num_layers=1)
    tables_d, ctx_d, qs_d, _, _ = G.step_metadata(wl)
    q = torch.zeros(100, 32, 128, dtype=torch.float16, device="cuda")
    out = torch.zeros_like(q)
    p.prefill_attn(0, q, qs_d, tables_d, ctx_d, 64, G.SCALE, out)          # q_len 100 above max_q_len 64
    st, flags = p.get_status()
    assert st == pkv.PKV_E_DEVICE and flags & pkv.PKV_DEV_BAD_QLEN
    bad = tables_d.clone()
    bad[0, 3] = wl.num_blocks + 1
    p.prefill_attn(0, q, qs_d, bad, ctx_d, 100, G.SCALE, out)
    st, flags = p.get_status()
    assert st == pkv.PKV_E_DEVICE and flags & pkv.PKV_DEV_BAD_BLOCK
    assert not out.any()                                                  # nothing was written
