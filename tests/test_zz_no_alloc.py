"""pkv_decode_attn_noalloc: decode attention for callers that cannot allocate.

Some callers cannot call cudaMalloc on the decode path (a plug-in whose host
process owns all device memory, a serving loop that forbids allocation after
start-up). This entry point uses a 16 MiB scratch array built into the
library instead of a caller workspace. The test calls it through the C ABI
twice in a row, on different inputs so the second call finds the first
call's leftovers in the shared scratch, and compares each result with the
workspace-taking pkv_decode_attn on the same inputs, within the parity
tolerance the other tests use. It also checks that a request too large for
the built-in scratch is refused before launch. This file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return G.lib()


def _case(seed, num_seqs, max_ctx):
    wl = workloads.random_step(seed, num_seqs=num_seqs, max_ctx=max_ctx, min_ctx=600, num_blocks=2048, num_layers=2)
    q, _, _ = G.new_token_inputs(wl, 1)
    tables_d, ctx_d, _, _, _ = G.step_metadata(wl)
    return q, tables_d, ctx_d


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row(pkv):
    pool_t = G.device_pool(2048, 2, 32, seed=31)
    pool = pkv.Pool(pool_t, 2048, num_layers=2)
    lib = pkv.load()
    stream = torch.cuda.current_stream().cuda_stream
    for seed, rows, max_ctx in ((41, 11, 3000), (42, 7, 2200)):
        q, tables_d, ctx_d = _case(seed, rows, max_ctx)
        assert tables_d.shape[1] * 16 > 1024, "the case must use more than one partition (the scratch)"
        ref = torch.empty_like(q)
        ws = torch.empty(pool.decode_workspace_bytes(rows, tables_d.shape[1]), dtype=torch.uint8, device="cuda")
        pool.decode_attn(1, q, tables_d, ctx_d, G.SCALE, ref, ws)
        out = torch.full_like(q, float("nan"))
        st = lib.pkv_decode_attn_noalloc(pool.handle, 1, q.data_ptr(), tables_d.data_ptr(), tables_d.shape[1],
                                         ctx_d.data_ptr(), rows, ctypes.c_float(G.SCALE), out.data_ptr(), stream)
        assert st == pkv.PKV_OK, lib.pkv_last_error_string()
        assert pool.get_status() == (pkv.PKV_OK, 0)
        G.assert_close(out, G.to_f64(ref), f"no-alloc decode, seed {seed}")


def test_noalloc_refuses_requests_beyond_its_scratch(pkv):
    pool_t = G.device_pool(64, 1, 32, seed=32)
    pool = pkv.Pool(pool_t, 64, num_layers=1)
    lib = pkv.load()
    rows, width = 1000, 1000          # ~1000 x 32 x 32 partials: far above 16 MiB
    st = lib.pkv_decode_attn_noalloc(pool.handle, 0, 16, 16, width, 16, rows, ctypes.c_float(G.SCALE), 16, None)
    assert st == pkv.PKV_E_INVALID
    assert b"scratch" in lib.pkv_last_error_string()
    assert pool.get_status() == (pkv.PKV_OK, 0)
