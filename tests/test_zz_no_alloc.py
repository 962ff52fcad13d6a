"""pkv_decode_attn_noalloc: decode attention for callers that cannot allocate.

Some callers cannot call cudaMalloc on the decode path: a plug-in whose host
process owns all device memory through its own allocator, or a serving loop
that forbids allocation after start-up because the call can synchronise the
device. This entry point uses a 16 MiB scratch array built into the library
instead of a caller workspace.

The test calls it through the C ABI twice in a row on each kind of pool the
decode path serves (FP16 with one query head per K/V head, FP16 with 8 K/V
heads serving 32 query heads, 8-bit codes), on different inputs so the
second call finds the first call's leftovers in the shared scratch. Each
result is compared with the workspace-taking pkv_decode_attn on the same
inputs and with the oracle, within the parity tolerance the other tests use.
It also checks that a request too large for the built-in scratch is refused
before launch. This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import _gpu as G

pytestmark = pytest.mark.gpu

CASES = ((41, 11, 3000), (42, 7, 2200))          # (seed, rows, longest context): several partitions each
KINDS = {"fp16_mha": (32, 32, "fp16"), "fp16_gqa": (8, 32, "fp16"), "int8_mha": (32, 32, "int8")}


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return G.lib()


def _pool(pkv, kind, num_blocks, layers):
    heads, q_heads, dtype = KINDS[kind]
    if dtype == "int8":
        t = G.device_pool_i8(num_blocks, layers, heads, seed=31)
        host = t.detach().cpu().numpy().reshape(-1).copy()
    else:
        t = G.device_pool(num_blocks, layers, heads, seed=31)
        host = G.to_bits(t).reshape(t.shape).copy()
    pool = pkv.Pool(t, num_blocks, num_layers=layers, num_heads=heads, num_q_heads=q_heads, dtype=dtype)
    g = oracle.geom(num_blocks, layers, heads, dtype=oracle.INT8 if dtype == "int8" else oracle.FP16,
                    num_q_heads=q_heads)
    return t, pool, host, g


@pytest.mark.parametrize("kind", sorted(KINDS))
def test_noalloc_matches_workspace_decode_and_oracle_on_two_calls_in_a_row(pkv, kind):
    layers, layer = 2, 1
    num_blocks = max(rows * -(-ctx // 16) for _, rows, ctx in CASES) + 16
    _, pool, host, g = _pool(pkv, kind, num_blocks, layers)
    q_heads = KINDS[kind][1]
    lib = pkv.load()
    stream = torch.cuda.current_stream().cuda_stream
    for seed, rows, max_ctx in CASES:
        wl = workloads.random_step(seed, num_seqs=rows, max_ctx=max_ctx, min_ctx=600, num_blocks=num_blocks,
                                   num_layers=layers)
        q = workloads.normal_fp16((rows, q_heads, 128), workloads.value_seed(seed, "q", layer)).cuda()
        tables_d, ctx_d = torch.from_numpy(wl.block_tables).cuda(), torch.from_numpy(wl.ctx_lens).cuda()
        assert wl.max_blocks * 16 > 1024, "the case must use more than one partition (the scratch)"
        ref = torch.empty_like(q)
        ws = torch.empty(pool.decode_workspace_bytes(rows, wl.max_blocks), dtype=torch.uint8, device="cuda")
        pool.decode_attn(layer, q, tables_d, ctx_d, G.SCALE, ref, ws)
        out = torch.full_like(q, float("nan"))
        st = lib.pkv_decode_attn_noalloc(pool.handle, layer, q.data_ptr(), tables_d.data_ptr(), wl.max_blocks,
                                         ctx_d.data_ptr(), rows, ctypes.c_float(G.SCALE), out.data_ptr(), stream)
        assert st == pkv.PKV_OK, lib.pkv_last_error_string()
        assert pool.get_status() == (pkv.PKV_OK, 0)
        G.assert_close(out, G.to_f64(ref), f"{kind}: no-alloc decode against pkv_decode_attn, seed {seed}")
        want, _ = oracle.decode_attn(host, g, layer, G.to_bits(q), wl.block_tables, wl.ctx_lens, G.SCALE)
        G.assert_close(out, want, f"{kind}: no-alloc decode against the oracle, seed {seed}")


def test_noalloc_refuses_requests_beyond_its_scratch(pkv):
    pool_t = G.device_pool(64, 1, 32, seed=32)
    pool = pkv.Pool(pool_t, 64, num_layers=1)
    lib = pkv.load()
    rows, width = 1000, 1000          # ~1000 x 32 x 16 partials: far above 16 MiB
    st = lib.pkv_decode_attn_noalloc(pool.handle, 0, 16, 16, width, 16, rows, ctypes.c_float(G.SCALE), 16, None)
    assert st == pkv.PKV_E_INVALID
    assert b"scratch" in lib.pkv_last_error_string()
    assert pool.get_status() == (pkv.PKV_OK, 0)
