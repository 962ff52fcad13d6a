"""GPU parity of cascade decode (rows sharing a prompt prefix read the shared blocks once per group)
against the oracle, and against the plain decode kernel, on the shared-prefix workload shape.
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


def _groups_wl(seed, sizes, prefix_blocks, max_private=120, num_layers=1):
    """Rows in consecutive groups; group i's rows share prefix_blocks[i] blocks, then 1..max_private own tokens."""
    rng = np.random.default_rng(seed)
    rows, ctx = [], []
    nb_total = sum(prefix_blocks) + sum(sizes) * (-(-max_private // 16)) + 16
    perm = rng.permutation(nb_total).astype(np.int32)
    cur = 0
    width = max(prefix_blocks) + (-(-max_private // 16)) + 1
    for n, pb in zip(sizes, prefix_blocks):
        shared = perm[cur:cur + pb]
        cur += pb
        for _ in range(n):
            u = int(rng.integers(1, max_private + 1))
            own = -(-u // 16)
            t = np.full(width, -1, np.int32)
            t[:pb] = shared
            t[pb:pb + own] = perm[cur:cur + own]
            cur += own
            rows.append(t)
            ctx.append(pb * 16 + u)
    tables = np.stack(rows)
    ctx = np.array(ctx, np.int32)
    return workloads.Workload(f"groups{seed}", num_layers, nb_total, tables, ctx, np.ones(len(ctx), np.int32), seed)


def run_cascade(pkv, wl, partition, check_plain=True, heads=32, q_heads=None, dtype="fp16"):
    H, hq = heads, q_heads or heads
    i8 = dtype == "int8"
    if i8:
        pool = G.device_pool_i8(wl.num_blocks, wl.num_layers, H, seed=wl.seed)
        host = pool.detach().cpu().numpy().reshape(-1).copy()
    else:
        pool = G.device_pool(wl.num_blocks, wl.num_layers, H, seed=wl.seed)
        host = G.to_bits(pool).reshape(pool.shape).copy()
    p = pkv.Pool(pool, wl.num_blocks, num_layers=wl.num_layers, num_heads=H, partition_tokens=partition,
                 num_q_heads=hq, dtype=dtype)
    tables_d, ctx_d, _, slots_d, slots = G.step_metadata(wl)
    T = wl.num_tokens
    q = workloads.normal_fp16((T, hq, 128), workloads.value_seed(wl.seed, "q")).cuda()
    k = workloads.normal_fp16((T, H, 128), workloads.value_seed(wl.seed, "k")).cuda()
    v = workloads.normal_fp16((T, H, 128), workloads.value_seed(wl.seed, "v")).cuda()
    p.kv_append(0, k, v, slots_d)
    g = oracle.geom(wl.num_blocks, wl.num_layers, H, num_q_heads=hq, dtype=oracle.INT8 if i8 else oracle.FP16)
    assert oracle.kv_append(host, g, 0, G.to_bits(k), G.to_bits(v), slots) == -1
    gs, gb, widest = pkv.cascade_groups(wl.block_tables, wl.ctx_lens)
    groups = (torch.from_numpy(gs).cuda(), torch.from_numpy(gb).cuda(), widest)
    ws = torch.empty(max(p.decode_cascade_workspace_bytes(wl.num_seqs, wl.max_blocks), 256), dtype=torch.uint8,
                     device="cuda")
    assert p.decode_cascade_workspace_bytes(wl.num_seqs, wl.max_blocks) >= p.decode_workspace_bytes(wl.num_seqs,
                                                                                                     wl.max_blocks)
    out = torch.full_like(q, float("nan"))
    p.decode_attn_cascade(0, q, tables_d, ctx_d, groups, G.SCALE, out, ws)
    assert p.get_status() == (pkv.PKV_OK, 0)
    ref, _ = oracle.decode_attn(host, g, 0, G.to_bits(q), wl.block_tables, wl.ctx_lens, G.SCALE)
    what = f"cascade, partition {partition}, {hq} query / {H} K/V heads, {dtype}"
    G.assert_close(out, ref, what)
    again = torch.full_like(q, float("nan"))
    p.decode_attn_cascade(0, q, tables_d, ctx_d, groups, G.SCALE, again, ws)
    assert torch.equal(out, again), what                # deterministic for a given grouping
    if check_plain:
        plain = torch.empty_like(q)
        p.decode_attn(0, q, tables_d, ctx_d, G.SCALE, plain, ws)   # the counters were left at zero
        assert p.get_status() == (pkv.PKV_OK, 0)
        G.assert_close(plain, ref, "plain decode after " + what)
    return gs, gb


@pytest.mark.parametrize("partition", [64, 256, 1024])
def test_cascade_groups_of_many_sizes(pkv, partition):
    # groups of 1, 5, 16, 17 (two row slices) and 40 rows; shared prefixes of 3 to 70 blocks
    wl = _groups_wl(1, [1, 5, 16, 17, 40], [3, 70, 20, 5, 64])
    gs, gb = run_cascade(pkv, wl, partition)
    assert list(np.diff(gs)) == [1, 5, 16, 17, 40] and list(gb) == [0, 70, 20, 5, 64]


def test_cascade_shared_prefix_config(pkv):
    # the shared-prefix workload's shape: 64 rows over 125 shared blocks + 1..300 private tokens (one layer)
    wl = workloads.shared_prefix_decode(0, num_layers=1, num_blocks=1500)
    gs, gb = run_cascade(pkv, wl, 0)
    assert list(gb) == [125] and list(gs) == [0, 64]


def test_cascade_without_sharing_equals_plain_decode(pkv):
    wl = workloads.random_step(3, num_seqs=7, max_ctx=900, num_blocks=500, num_layers=1)
    gs, gb = run_cascade(pkv, wl, 64)
    assert not gb.any()


def test_cascade_refuses_bad_groups_and_pools(pkv):
    wl = _groups_wl(4, [4], [10])
    pool = G.device_pool(wl.num_blocks, 1, 32, seed=4)
    p = pkv.Pool(pool, wl.num_blocks, num_layers=1)
    tables_d, ctx_d, _, _, _ = G.step_metadata(wl)
    q = torch.zeros(4, 32, 128, dtype=torch.float16, device="cuda")
    ws = torch.empty(p.decode_cascade_workspace_bytes(4, wl.max_blocks), dtype=torch.uint8, device="cuda")
    small = torch.empty(p.decode_workspace_bytes(4, wl.max_blocks), dtype=torch.uint8, device="cuda")
    ok = (torch.tensor([0, 4], dtype=torch.int32, device="cuda"), torch.tensor([10], dtype=torch.int32, device="cuda"),
          4)
    with pytest.raises(pkv.PkvError):                      # the plain decode's workspace is one slot short
        p.decode_attn_cascade(0, q, tables_d, ctx_d, ok, G.SCALE, q, small)
    bad = (torch.tensor([0, 4], dtype=torch.int32, device="cuda"), torch.tensor([10], dtype=torch.int32, device="cuda"),
           9)                                              # max_group_rows above num_seqs
    with pytest.raises(pkv.PkvError):
        p.decode_attn_cascade(0, q, tables_d, ctx_d, bad, G.SCALE, q, ws)
    empty = (torch.tensor([0, 4], dtype=torch.int32, device="cuda"),
             torch.tensor([10], dtype=torch.int32, device="cuda"), 0)          # max_group_rows below 1
    with pytest.raises(pkv.PkvError):
        p.decode_attn_cascade(0, q, tables_d, ctx_d, empty, G.SCALE, q, ws)


# Grouped query heads and 8-bit pools: (K/V heads, query heads, element type). A shared-prefix CTA holds 16 query
# rows: 4 rows x 4 heads (G = 4), 2 rows x 8 heads (MQA with 8 query heads), 1 row x 12 heads (G = 12), one row's
# 16-head slice of a 32-head group (G = 32, two slices); 8-bit pools with 1, 4 and 7 query heads per K/V head
# (G = 7: 2 rows x 7 heads in a shared-prefix CTA, an odd column count in the private keys' transposed form).
KINDS = [(8, 32, "fp16"), (1, 8, "fp16"), (4, 48, "fp16"), (2, 64, "fp16"), (32, 32, "int8"), (8, 32, "int8"),
         (2, 14, "int8")]


@pytest.mark.parametrize("heads,q_heads,dtype", KINDS)
@pytest.mark.parametrize("partition", [64, 1024])
def test_cascade_grouped_heads_and_8bit_pools(pkv, heads, q_heads, dtype, partition):
    wl = _groups_wl(5, [1, 6, 9, 17], [4, 40, 9, 66])
    gs, gb = run_cascade(pkv, wl, partition, heads=heads, q_heads=q_heads, dtype=dtype)
    assert list(np.diff(gs)) == [1, 6, 9, 17] and list(gb) == [0, 40, 9, 66]


@pytest.mark.parametrize("heads,q_heads,dtype", [(8, 32, "fp16"), (32, 32, "int8"), (8, 32, "int8")])
def test_cascade_shared_prefix_config_grouped_and_8bit(pkv, heads, q_heads, dtype):
    # the shared-prefix workload's shape (64 rows over 125 shared blocks) with 8 K/V heads and over an 8-bit pool
    wl = workloads.shared_prefix_decode(0, num_layers=1, num_blocks=1500)
    gs, gb = run_cascade(pkv, wl, 0, heads=heads, q_heads=q_heads, dtype=dtype)
    assert list(gb) == [125] and list(gs) == [0, 64]


@pytest.mark.parametrize("heads,q_heads,dtype", [(32, 32, "fp16"), (32, 32, "int8")])
def test_cascade_back_to_back_calls_are_bit_identical(pkv, heads, q_heads, dtype):
    # The shared-prefix and private-key launches run side by side (FP16 with one query head per K/V head, and
    # 8-bit pools), and whichever partial of a row arrives last merges it. Twelve calls back to back on one
    # stream, reusing one workspace: every output must be bit-identical (the merge is the same arithmetic
    # whichever launch does it), and no call may see the previous call's launches still running (its counter
    # clear would otherwise race their arrivals: rows merged twice, or never).
    wl = workloads.shared_prefix_decode(1, num_layers=1, num_blocks=1500)
    i8 = dtype == "int8"
    pool = (G.device_pool_i8 if i8 else G.device_pool)(wl.num_blocks, 1, heads, seed=wl.seed)
    p = pkv.Pool(pool, wl.num_blocks, num_layers=1, num_heads=heads, num_q_heads=q_heads, dtype=dtype)
    tables_d, ctx_d, _, _, _ = G.step_metadata(wl)
    q = workloads.normal_fp16((wl.num_tokens, q_heads, 128), workloads.value_seed(wl.seed, "q")).cuda()
    gs, gb, widest = pkv.cascade_groups(wl.block_tables, wl.ctx_lens)
    groups = (torch.from_numpy(gs).cuda(), torch.from_numpy(gb).cuda(), widest)
    ws = torch.empty(max(p.decode_cascade_workspace_bytes(wl.num_seqs, wl.max_blocks), 256), dtype=torch.uint8,
                     device="cuda")
    outs = [torch.full_like(q, float("nan")) for _ in range(12)]
    for o in outs:
        p.decode_attn_cascade(0, q, tables_d, ctx_d, groups, G.SCALE, o, ws)
    assert p.get_status() == (pkv.PKV_OK, 0)
    assert not torch.isnan(outs[0]).any()
    for i, o in enumerate(outs[1:], 1):
        assert torch.equal(o, outs[0]), f"call {i} differs from call 0"
    plain = torch.empty_like(q)
    p.decode_attn(0, q, tables_d, ctx_d, G.SCALE, plain, ws)  # the counters were left at zero
    assert p.get_status() == (pkv.PKV_OK, 0)
    # both lie within the attention tolerance of the same exact result, so within twice it of each other
    d, ref = (plain.double() - outs[0].double()).abs(), plain.double().abs()
    assert bool((d <= 2 * (2e-3 + 1e-2 * ref)).all()), d.max().item()
