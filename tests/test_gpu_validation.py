"""Refusals of the device calls on the host: bad step sizes, layer ranges, strides, alignment and workspace
sizes come back as PKV_E_INVALID before anything is launched, so the pool, the outputs and the device status
word stay as they were."""
import numpy as np
import pytest
import torch

import workloads
from tests import _gpu as G

pytestmark = pytest.mark.gpu
H = 32


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pkv = G.lib()
    wl = workloads.random_step(5, num_seqs=4, max_ctx=100, num_blocks=64, num_layers=2, prefill_rows=1, max_q=20)
    pool_t = G.device_pool(wl.num_blocks, 2, H, seed=5)
    p = pkv.Pool(pool_t, wl.num_blocks, num_layers=2, partition_tokens=64)
    tables_d, ctx_d, qs_d, slots_d, _ = G.step_metadata(wl)
    T = wl.num_tokens
    q = torch.zeros(2, T, H, 128, dtype=torch.float16, device="cuda")
    k, v = torch.zeros_like(q), torch.zeros_like(q)
    out = torch.full_like(q, 7.0)
    return dict(pkv=pkv, wl=wl, pool_t=pool_t, p=p, tables=tables_d, ctx=ctx_d, qs=qs_d, slots=slots_d, q=q, k=k,
                v=v, out=out)


def _step(e, **over):
    wl = e["wl"]
    T, B = wl.num_tokens, wl.num_decode
    kw = dict(num_decode=B, num_prefill=wl.num_seqs - B, num_tokens=T, max_q_len=int(wl.q_lens.max()),
              max_blocks=wl.max_blocks, first_layer=0, num_layers=2, scale=G.SCALE, block_tables=e["tables"],
              ctx_lens=e["ctx"], q_start_loc=e["qs"], slot_mapping=e["slots"], q=e["q"], k=e["k"], v=e["v"],
              out=e["out"], q_layer_stride=T * H * 128, k_layer_stride=T * H * 128, v_layer_stride=T * H * 128,
              out_layer_stride=T * H * 128)
    kw.update(over)
    return e["pkv"].make_step_desc(**kw)


def _refused(e, fn):
    pkv = e["pkv"]
    before = G.to_bits(e["pool_t"]).copy()
    with pytest.raises(pkv.PkvError) as err:
        fn()
    assert err.value.status == pkv.PKV_E_INVALID
    torch.cuda.synchronize()
    assert np.array_equal(G.to_bits(e["pool_t"]), before)           # nothing appended
    assert bool((e["out"] == 7.0).all())                             # nothing written
    assert e["p"].get_status() == (pkv.PKV_OK, 0)                    # nothing launched that failed


def test_step_refusals(env):
    e, p = env, env["p"]
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    _refused(e, lambda: p.step(_step(e, max_q_len=0), ws))                   # prefill rows need max_q_len >= 1
    _refused(e, lambda: p.step(_step(e, num_layers=3), ws))                  # layers past the pool's
    _refused(e, lambda: p.step(_step(e, first_layer=-1), ws))
    _refused(e, lambda: p.step(_step(e, q_layer_stride=e["wl"].num_tokens * H * 128 + 4), ws))  # not x8
    _refused(e, lambda: p.step(_step(e, num_tokens=e["wl"].num_decode + e["wl"].num_seqs - e["wl"].num_decode - 1),
                               ws))                                          # fewer tokens than rows
    _refused(e, lambda: p.step(_step(e, num_prefill=0, num_tokens=e["wl"].num_tokens), ws))  # decode-only, T != B
    _refused(e, lambda: p.step(_step(e, block_tables=None), ws))             # NULL array


def test_call_refusals(env):
    e, p = env, env["p"]
    wl = e["wl"]
    B = wl.num_decode
    q1 = e["q"][0]
    # q or out not 16-byte aligned: a view 2 bytes into the buffer
    flat = torch.zeros(q1.numel() + 8, dtype=torch.float16, device="cuda")
    q_off = flat[1:1 + q1.numel()].view(q1.shape)
    _refused(e, lambda: p.prefill_attn(0, q_off, e["qs"][B:], e["tables"][B:], e["ctx"][B:], int(wl.q_lens.max()),
                                       G.SCALE, e["out"][0]))
    _refused(e, lambda: p.kv_append(0, q_off, e["v"][0], e["slots"]))        # k not 16-byte aligned
    # a decode workspace below what the pool's 64-token partitions need
    need = p.decode_workspace_bytes(B, wl.max_blocks)
    assert need > 256
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    _refused(e, lambda: p.decode_attn(0, q1[:B].contiguous(), e["tables"][:B], e["ctx"][:B], G.SCALE,
                                      e["out"][0][:B], small))
    _refused(e, lambda: p.decode_attn(2, q1[:B].contiguous(), e["tables"][:B], e["ctx"][:B], G.SCALE,
                                      e["out"][0][:B], torch.empty(need, dtype=torch.uint8, device="cuda")))  # layer 2 of 2
