"""Parity at full size for the grouped-head, 8-bit (decode and chunked prefill) and cascade paths, in the
launch configuration bench.py times (pkv_step over 32 layers; cascade: kv_append + pkv_decode_attn_cascade per
layer).

Sampled (layer, row) outputs are checked against the oracle, which gets host copies of the row's blocks
taken before the step plus its own append of the row's new token; every new token's stored K/V (FP16
bits, or INT8 codes and scales) is checked in every layer.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _gpu as G

pytestmark = pytest.mark.gpu
L = workloads.NUM_LAYERS


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return G.lib()


def _inputs(T, hq, h, seed):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    q = torch.randn((L, T, hq, 128), generator=gen, device="cuda").half()
    k = torch.randn((L, T, h, 128), generator=gen, device="cuda").half()
    v = torch.randn((L, T, h, 128), generator=gen, device="cuda").half()
    return q, k, v


def _step_desc(pkv, wl, tables_d, ctx_d, qs_d, slots_d, q, k, v, out, hq, h):
    T = wl.num_tokens
    return pkv.make_step_desc(num_decode=T, num_prefill=0, num_tokens=T, max_q_len=0, max_blocks=wl.max_blocks,
                              first_layer=0, num_layers=L, scale=G.SCALE, block_tables=tables_d, ctx_lens=ctx_d,
                              q_start_loc=qs_d, slot_mapping=slots_d, q=q, k=k, v=v, out=out,
                              q_layer_stride=T * hq * 128, k_layer_stride=T * h * 128, v_layer_stride=T * h * 128,
                              out_layer_stride=T * hq * 128)


def _check_rows(wl, g, copies, qb, kb, vb, out, hq):
    for (l, r), mini in copies.items():
        ctx = int(wl.ctx_lens[r])
        nblk = -(-ctx // 16)
        gm = oracle.geom(nblk, 1, g.num_heads, num_q_heads=hq, dtype=g.dtype)
        pos = np.array([ctx - 1], np.int64)
        assert oracle.kv_append(mini, gm, 0, kb[l, r][None], vb[l, r][None], pos) == -1
        ref, _ = oracle.decode_attn(mini, gm, 0, qb[l, r][None], np.arange(nblk, dtype=np.int32)[None],
                                    np.array([ctx], np.int32), G.SCALE)
        G.assert_close(out[l, r], ref[0], f"{wl.name} layer {l} row {r}")


def test_full_gqa_decode(pkv):
    wl = workloads.gqa_decode(0)
    H, HQ, N = wl.num_heads, wl.q_heads, wl.num_blocks
    pool_t = torch.empty(workloads.pool_shape(N, L, H), dtype=torch.float16, device="cuda")
    workloads.fill_normal_fp16_(pool_t, workloads.value_seed(0, "pool"))
    # the pool's partition length bench.py uses for this workload: one 4,096-token partition per 2,300-token row
    p = pkv.Pool(pool_t, N, num_layers=L, num_heads=H, num_q_heads=HQ, partition_tokens=4096)
    tables_d, ctx_d, qs_d, slots_d, slots = G.step_metadata(wl)
    q, k, v = _inputs(wl.num_tokens, HQ, H, 5)
    out = torch.full_like(q, float("nan"))
    samples = [(0, 0), (7, 13), (19, 31), (31, 5)]
    copies = {}
    for l, r in samples:
        ids = torch.from_numpy(wl.block_tables[r, :144].astype(np.int64)).cuda()
        sub = pool_t.index_select(0, ids)[:, l:l + 1].contiguous()
        copies[(l, r)] = G.to_bits(sub).reshape(sub.shape)
    sd = _step_desc(pkv, wl, tables_d, ctx_d, qs_d, slots_d, q, k, v, out, HQ, H)
    ws = torch.empty(max(p.step_workspace_bytes(sd), 256), dtype=torch.uint8, device="cuda")
    p.step(sd, ws)
    assert p.get_status() == (pkv.PKV_OK, 0)
    s = torch.from_numpy(slots).cuda()
    for l in range(L):
        assert torch.equal(pool_t[s // 16, l, 0, :, s % 16, :], k[l]) and \
            torch.equal(pool_t[s // 16, l, 1, :, s % 16, :], v[l]), f"append differs at layer {l}"
    g = oracle.geom(N, L, H, num_q_heads=HQ)
    _check_rows(wl, g, copies, G.to_bits(q), G.to_bits(k), G.to_bits(v), out, HQ)
    del pool_t
    torch.cuda.empty_cache()


def test_full_int8_average_decode(pkv):
    wl = workloads.average_decode(0)
    H, N = wl.num_heads, wl.num_blocks
    pool_t = torch.empty(pkv.Pool.bytes_needed(N, L, H, "int8"), dtype=torch.uint8, device="cuda")
    workloads.fill_int8_tiles_(pool_t, workloads.value_seed(0, "pool"))
    tiles = pool_t.view(N, L, 2, H, 2112)
    p = pkv.Pool(pool_t, N, num_layers=L, num_heads=H, dtype="int8")
    tables_d, ctx_d, qs_d, slots_d, slots = G.step_metadata(wl)
    q, k, v = _inputs(wl.num_tokens, H, H, 6)
    out = torch.full_like(q, float("nan"))
    samples = [(0, int(np.argmax(wl.ctx_lens))), (11, 3), (23, 17), (31, int(np.argmin(wl.ctx_lens)))]
    copies = {}
    for l, r in samples:
        nb = -(-int(wl.ctx_lens[r]) // 16)
        ids = torch.from_numpy(wl.block_tables[r, :nb].astype(np.int64)).cuda()
        copies[(l, r)] = tiles.index_select(0, ids)[:, l].contiguous().cpu().numpy().reshape(-1).copy()
    sd = _step_desc(pkv, wl, tables_d, ctx_d, qs_d, slots_d, q, k, v, out, H, H)
    ws = torch.empty(max(p.step_workspace_bytes(sd), 256), dtype=torch.uint8, device="cuda")
    p.step(sd, ws)
    assert p.get_status() == (pkv.PKV_OK, 0)
    # every new token's codes and scales, every layer, against the oracle's quantiser
    blk, t = slots // 16, slots % 16
    kb, vb = G.to_bits(k), G.to_bits(v)
    for l in range(L):
        got = tiles[torch.from_numpy(blk).cuda(), l].cpu().numpy()         # [T, 2, H, 2112]
        for i in range(wl.num_tokens):
            for kv, src in ((0, kb), (1, vb)):
                for h in range(0, H, 7):
                    codes, scale = oracle.i8_quantize_row(src[l, i, h])
                    row = got[i, kv, h]
                    assert np.array_equal(row[t[i] * 128:(t[i] + 1) * 128].view(np.int8), codes)
                    assert row[2048 + 4 * t[i]:2052 + 4 * t[i]].view(np.float32)[0] == scale
    g = oracle.geom(N, L, H, dtype=oracle.INT8)
    _check_rows(wl, g, copies, G.to_bits(q), kb, vb, out, H)
    del pool_t, tiles
    torch.cuda.empty_cache()


def test_full_shared_prefix_cascade(pkv):
    wl = workloads.shared_prefix_decode(0)
    H, N = wl.num_heads, wl.num_blocks
    pool_t = torch.empty(workloads.pool_shape(N, L, H), dtype=torch.float16, device="cuda")
    workloads.fill_normal_fp16_(pool_t, workloads.value_seed(0, "pool"))
    p = pkv.Pool(pool_t, N, num_layers=L, num_heads=H)
    tables_d, ctx_d, qs_d, slots_d, slots = G.step_metadata(wl)
    q, k, v = _inputs(wl.num_tokens, H, H, 7)
    out = torch.full_like(q, float("nan"))
    samples = [(0, 0), (9, 40), (30, 63)]
    copies = {}
    for l, r in samples:
        nb = -(-int(wl.ctx_lens[r]) // 16)
        ids = torch.from_numpy(wl.block_tables[r, :nb].astype(np.int64)).cuda()
        sub = pool_t.index_select(0, ids)[:, l:l + 1].contiguous()
        copies[(l, r)] = G.to_bits(sub).reshape(sub.shape)
    gs, gb, widest = pkv.cascade_groups(wl.block_tables, wl.ctx_lens)
    assert list(gb) == [125]
    groups = (torch.from_numpy(gs).cuda(), torch.from_numpy(gb).cuda(), widest)
    ws = torch.empty(p.decode_cascade_workspace_bytes(wl.num_seqs, wl.max_blocks), dtype=torch.uint8, device="cuda")
    for l in range(L):
        p.kv_append(l, k[l], v[l], slots_d)
        p.decode_attn_cascade(l, q[l], tables_d, ctx_d, groups, G.SCALE, out[l], ws)
    assert p.get_status() == (pkv.PKV_OK, 0)
    g = oracle.geom(N, L, H)
    _check_rows(wl, g, copies, G.to_bits(q), G.to_bits(k), G.to_bits(v), out, H)
    del pool_t
    torch.cuda.empty_cache()


def test_full_int8_mixed_chunked_prefill(pkv):
    """The 8-chunk schedule of a 4,000-token prompt next to 31 decode rows over an 8-bit pool (30.9 GB),
    through pkv_step as bench.py times it: after every chunk the prompt's stored codes and scales equal the
    oracle's own append; sampled prompt rows (chunks 0, 1, 6, 7) and decode rows against the oracle."""
    first = workloads.mixed_prefill(0)
    H, N = first.num_heads, first.num_blocks
    nchunks = first.meta["num_chunks"]
    P = first.num_seqs - 1                    # the prompt row
    pool_t = torch.empty(pkv.Pool.bytes_needed(N, L, H, "int8"), dtype=torch.uint8, device="cuda")
    workloads.fill_int8_tiles_(pool_t, workloads.value_seed(0, "pool"))
    tiles = pool_t.view(N, L, 2, H, 2112)
    p = pkv.Pool(pool_t, N, num_layers=L, num_heads=H, dtype="int8")
    layers, dec_rows = (0, 31), (0, 30)
    prompt_nb = -(-first.meta["prompt_len"] // 16)
    prompt_ids = torch.from_numpy(first.block_tables[P, :prompt_nb].astype(np.int64)).cuda()
    mini = {l: tiles.index_select(0, prompt_ids)[:, l].contiguous().cpu().numpy().reshape(-1).copy()
            for l in layers}
    dec_nb = {r: -(-int(first.ctx_lens[r] + nchunks - 1) // 16) for r in dec_rows}
    dec_mini = {(l, r): tiles.index_select(0, torch.from_numpy(first.block_tables[r, :dec_nb[r]].astype(
                np.int64)).cuda())[:, l].contiguous().cpu().numpy().reshape(-1).copy()
                for l in layers for r in dec_rows}
    g = oracle.geom(prompt_nb, 1, H, dtype=oracle.INT8)
    table = np.arange(prompt_nb, dtype=np.int32)[None]
    rng = np.random.default_rng(9)
    for c in range(nchunks):
        wl = workloads.mixed_prefill(c)
        T, B = wl.num_tokens, wl.num_decode
        start, end = wl.meta["chunk_start"], wl.meta["chunk_end"]
        tables_d, ctx_d, qs_d, slots_d, slots = G.step_metadata(wl)
        q, k, v = _inputs(T, H, H, 40 + c)
        out = torch.full_like(q, float("nan"))
        sd = pkv.make_step_desc(num_decode=B, num_prefill=1, num_tokens=T, max_q_len=end - start,
                                max_blocks=wl.max_blocks, first_layer=0, num_layers=L, scale=G.SCALE,
                                block_tables=tables_d, ctx_lens=ctx_d, q_start_loc=qs_d, slot_mapping=slots_d,
                                q=q, k=k, v=v, out=out, q_layer_stride=T * H * 128, k_layer_stride=T * H * 128,
                                v_layer_stride=T * H * 128, out_layer_stride=T * H * 128)
        ws = torch.empty(max(p.step_workspace_bytes(sd), 256), dtype=torch.uint8, device="cuda")
        p.step(sd, ws)
        assert p.get_status() == (pkv.PKV_OK, 0), f"chunk {c}"
        qb, kb, vb = G.to_bits(q), G.to_bits(k), G.to_bits(v)
        for l in layers:
            pos = np.arange(start, end, dtype=np.int64)
            assert oracle.kv_append(mini[l], g, 0, kb[l, B:], vb[l, B:], pos) == -1
            got = tiles.index_select(0, prompt_ids)[:, l].contiguous().cpu().numpy().reshape(-1)
            assert np.array_equal(got, mini[l]), f"chunk {c} layer {l}: prompt codes/scales differ"
            for r in dec_rows:
                ctx = int(wl.ctx_lens[r])
                gd = oracle.geom(dec_nb[r], 1, H, dtype=oracle.INT8)
                assert oracle.kv_append(dec_mini[(l, r)], gd, 0, kb[l, r][None], vb[l, r][None],
                                        np.array([ctx - 1], np.int64)) == -1
                ref, _ = oracle.decode_attn(dec_mini[(l, r)], gd, 0, qb[l, r][None],
                                            np.arange(dec_nb[r], dtype=np.int32)[None], np.array([ctx], np.int32),
                                            G.SCALE)
                G.assert_close(out[l, r], ref[0], f"chunk {c} layer {l} decode row {r}")
            if c not in (0, 1, 6, 7):
                continue
            picks = sorted(set([0, end - start - 1] + rng.integers(0, end - start, 14).tolist()))
            for i in picks:
                ref, _ = oracle.decode_attn(mini[l], g, 0, qb[l, B + i][None], table,
                                            np.array([start + i + 1], np.int32), G.SCALE)
                G.assert_close(out[l, B + i], ref[0], f"chunk {c} layer {l} prefill row {i}")
    del pool_t, tiles
    torch.cuda.empty_cache()
