"""Parity at the full workload sizes, in the launch configuration bench.py times.

A 60 GB pool (7,152 blocks x 32 layers x 32 heads x 128 dims FP16) is filled
on the GPU; each workload runs as pkv_step over all 32 layers. Checks:
  * kv_append: every new token's K/V row in every layer equals its input
    (bit-exact), and 4,096 random canary rows elsewhere are unchanged;
  * attention: sampled (layer, row) outputs against the oracle, which gets
    host copies of that row's blocks taken BEFORE the step plus its own
    kv_append of the step's new tokens — nothing the CUDA path produced.
Prefill rows are sampled one query at a time: the causal prefill row at
position p is the decode of that query over keys 0..p (pinned in the oracle
tests).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _gpu as G

pytestmark = pytest.mark.gpu

N_BLOCKS, L, H = workloads.POOL_BLOCKS, workloads.NUM_LAYERS, workloads.NUM_HEADS


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return G.lib()


@pytest.fixture(scope="module")
def big_pool(pkv):
    t = torch.empty(workloads.pool_shape(N_BLOCKS, L, H), dtype=torch.float16, device="cuda")
    workloads.fill_normal_fp16_(t, workloads.value_seed(0, "pool"))
    yield t
    del t
    torch.cuda.empty_cache()


def _layer_inputs(T, seed):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    return [torch.randn((L, T, H, 128), generator=gen, device="cuda").half() for _ in range(3)]


def _rows_copy(pool_t, table_row, nblk, layer):
    ids = torch.from_numpy(table_row[:nblk].astype(np.int64)).cuda()
    sub = pool_t.index_select(0, ids)[:, layer:layer + 1].contiguous()
    return G.to_bits(sub).reshape(sub.shape)


class Step:
    def __init__(self, pkv, pool, wl, seed):
        self.wl = wl
        self.tables_d, self.ctx_d, self.qs_d, self.slots_d, self.slots = G.step_metadata(wl)
        T = wl.num_tokens
        self.q, self.k, self.v = _layer_inputs(T, seed)
        self.out = torch.full_like(self.q, float("nan"))
        B = wl.num_decode
        self.desc = pkv.make_step_desc(
            num_decode=B, num_prefill=wl.num_seqs - B, num_tokens=T,
            max_q_len=int(wl.q_lens[B:].max()) if wl.num_seqs > B else 0, max_blocks=wl.max_blocks, first_layer=0,
            num_layers=L, scale=G.SCALE, block_tables=self.tables_d, ctx_lens=self.ctx_d, q_start_loc=self.qs_d,
            slot_mapping=self.slots_d, q=self.q, k=self.k, v=self.v, out=self.out, q_layer_stride=T * H * 128,
            k_layer_stride=T * H * 128, v_layer_stride=T * H * 128, out_layer_stride=T * H * 128)
        self.ws = torch.empty(max(pool.step_workspace_bytes(self.desc), 256), dtype=torch.uint8, device="cuda")

    def run(self, pkv, pool):
        pool.step(self.desc, self.ws)
        assert pool.get_status() == (pkv.PKV_OK, 0)

    def check_append(self, pool_t):
        s = torch.from_numpy(self.slots).cuda()
        blk, t = s // 16, s % 16
        for l in range(L):
            got_k = pool_t[blk, l, 0, :, t, :]
            got_v = pool_t[blk, l, 1, :, t, :]
            assert torch.equal(got_k, self.k[l]) and torch.equal(got_v, self.v[l]), f"append differs at layer {l}"


def _canaries(pool_t, exclude_slots, n=4096, seed=0):
    rng = np.random.default_rng(seed)
    written = set(int(x) for x in exclude_slots)
    picks = []
    while len(picks) < n:
        b, l, kv, h, t = (int(rng.integers(0, N_BLOCKS)), int(rng.integers(0, L)), int(rng.integers(0, 2)),
                          int(rng.integers(0, H)), int(rng.integers(0, 16)))
        if b * 16 + t not in written:
            picks.append((b, l, kv, h, t))
    idx = [torch.tensor(c, device="cuda") for c in zip(*picks)]
    return idx, pool_t[idx[0], idx[1], idx[2], idx[3], idx[4], :].clone()


def _oracle_row(mini, layer_tokens, q_row, ctx, nblk):
    """Oracle decode of one query over a row's blocks, after appending the row's new tokens.

    layer_tokens: list of (position, k bits [H,128], v bits [H,128])."""
    g = oracle.geom(nblk, 1, H)
    table = np.arange(nblk, dtype=np.int32)
    for pos, kb, vb in layer_tokens:
        assert oracle.kv_append(mini, g, 0, kb[None], vb[None], np.array([pos], np.int64)) == -1
    ref, _ = oracle.decode_attn(mini, g, 0, q_row[None], table[None], np.array([ctx], np.int32), G.SCALE)
    return ref[0]


def _decode_case(pkv, big_pool, wl, layers, rows, seed, partition=0):
    pool = pkv.Pool(big_pool, N_BLOCKS, num_layers=L, num_heads=H, partition_tokens=partition)
    st = Step(pkv, pool, wl, seed)
    copies = {}
    for l in layers:
        for r in rows:
            nb = -(-int(wl.ctx_lens[r]) // 16)
            copies[(l, r)] = _rows_copy(big_pool, wl.block_tables[r], nb, l)
    can_idx, can_before = _canaries(big_pool, st.slots, seed=seed)
    st.run(pkv, pool)
    st.check_append(big_pool)
    assert torch.equal(big_pool[can_idx[0], can_idx[1], can_idx[2], can_idx[3], can_idx[4], :], can_before)
    qb, kb, vb = G.to_bits(st.q), G.to_bits(st.k), G.to_bits(st.v)
    out = st.out
    for (l, r), mini in copies.items():
        ctx = int(wl.ctx_lens[r])
        ref = _oracle_row(mini, [(ctx - 1, kb[l, r], vb[l, r])], qb[l, r], ctx, mini.shape[0])
        G.assert_close(out[l, r], ref, f"{wl.name} layer {l} row {r}")


def test_full_average_decode(pkv, big_pool):
    wl = workloads.average_decode(0)
    # the pool's partition length bench.py uses for this workload (and the library default)
    for partition in (2048, 0):
        _decode_case(pkv, big_pool, wl, layers=(0, 13, 31), rows=range(wl.num_seqs), seed=101, partition=partition)


def test_full_long_decode(pkv, big_pool):
    wl = workloads.long_decode(0)
    _decode_case(pkv, big_pool, wl, layers=(0, 31), rows=(0, 6, 12), seed=102, partition=2048)


def test_full_shared_prefix_decode(pkv, big_pool):
    wl = workloads.shared_prefix_decode(0)
    _decode_case(pkv, big_pool, wl, layers=(0, 31), rows=(0, 9, 31, 50, 63), seed=103)


def test_full_mixed_chunked_prefill(pkv, big_pool):
    """The 8-chunk schedule of a 4,000-token prompt next to 31 decode rows, chunks in order on one pool."""
    pool = pkv.Pool(big_pool, N_BLOCKS, num_layers=L, num_heads=H)
    first = workloads.mixed_prefill(0)
    nchunks = first.meta["num_chunks"]
    P = first.num_seqs - 1                    # the prompt row
    layers = (0, 13, 31)
    prompt_nb = -(-first.meta["prompt_len"] // 16)
    prompt_copy = {l: _rows_copy(big_pool, first.block_tables[P], prompt_nb, l) for l in layers}
    dec_rows = (0, 15, 30)
    dec_copy = {}
    for l in layers:
        for r in dec_rows:
            nb = -(-int(first.ctx_lens[r] + nchunks - 1) // 16)
            dec_copy[(l, r)] = _rows_copy(big_pool, first.block_tables[r], nb, l)
    prompt_kv = {l: ([], [], []) for l in layers}   # positions, K rows, V rows appended so far
    dec_kv = {k: [] for k in dec_copy}
    rng = np.random.default_rng(7)
    g = oracle.geom(prompt_nb, 1, H)
    table = np.arange(prompt_nb, dtype=np.int32)[None]
    for c in range(nchunks):
        wl = workloads.mixed_prefill(c)
        st = Step(pkv, pool, wl, 200 + c)
        st.run(pkv, pool)
        st.check_append(big_pool)
        qb, kb, vb = G.to_bits(st.q), G.to_bits(st.k), G.to_bits(st.v)
        B = wl.num_decode
        start, end = wl.meta["chunk_start"], wl.meta["chunk_end"]
        for l in layers:
            pos_l, k_l, v_l = prompt_kv[l]
            pos_l.extend(range(start, end))
            k_l.append(kb[l, B:B + end - start])
            v_l.append(vb[l, B:B + end - start])
            for r in dec_rows:
                ctx = int(wl.ctx_lens[r])
                dec_kv[(l, r)].append((ctx - 1, kb[l, r], vb[l, r]))
                mini = dec_copy[(l, r)].copy()
                ref = _oracle_row(mini, dec_kv[(l, r)], qb[l, r], ctx, mini.shape[0])
                G.assert_close(st.out[l, r], ref, f"chunk {c} layer {l} decode row {r}")
            mini = prompt_copy[l].copy()
            assert oracle.kv_append(mini, g, 0, np.concatenate(k_l), np.concatenate(v_l),
                                    np.array(pos_l, np.int64)) == -1
            # every chunk: both rows at each 128-row query-tile boundary, the chunk's ends and 24 more
            n_q = end - start
            bounds = [x for b in range(0, n_q, 128) for x in (b, b + 127)]
            picks = sorted(set(x for x in [0, n_q - 1] + bounds + rng.integers(0, n_q, 24).tolist() if x < n_q))
            for i in picks:
                ref, _ = oracle.decode_attn(mini, g, 0, qb[l, B + i][None], table, np.array([start + i + 1], np.int32),
                                            G.SCALE)
                G.assert_close(st.out[l, B + i], ref[0], f"chunk {c} layer {l} prefill row {i}")
