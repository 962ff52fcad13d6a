"""Helpers shared by the GPU parity tests: seeded inputs on the device, the
oracle on host copies, and the FP16 tolerance check."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

SCALE = oracle.SCALE_FP32
# An element passes if |gpu - ref| <= ATOL + RTOL * |ref| (allclose convention),
# ref being the oracle's unrounded double result.
ATOL, RTOL = 2e-3, 1e-2


def lib():
    from paged_kv_cache_scatter_gb300 import build
    build.build()
    import paged_kv_cache_scatter_gb300 as pkv
    pkv.load()
    return pkv


def device_pool(num_blocks, num_layers, num_heads=32, seed=0, on_gpu_rng=False):
    shape = workloads.pool_shape(num_blocks, num_layers, num_heads)
    if on_gpu_rng:
        t = torch.empty(shape, dtype=torch.float16, device="cuda")
        workloads.fill_normal_fp16_(t, workloads.value_seed(seed, "pool"))
        return t
    return workloads.normal_fp16(shape, workloads.value_seed(seed, "pool")).cuda()


def device_pool_i8(num_blocks, num_layers, num_heads=32, seed=0):
    """An 8-bit pool with valid contents everywhere: codes uniform in [-127, 127], scales in [0.004, 0.03)
    (about what N(0,1) rows quantise to). Returns the device uint8 tensor [blocks, layers, 2, heads, 2112]."""
    rng = np.random.default_rng(workloads.value_seed(seed, "pool") + 7)
    tiles = np.empty((num_blocks, num_layers, 2, num_heads, 2112), np.uint8)
    tiles[..., :2048] = rng.integers(-127, 128, tiles[..., :2048].shape).astype(np.int8).view(np.uint8)
    scales = rng.uniform(0.004, 0.03, (num_blocks, num_layers, 2, num_heads, 16)).astype(np.float32)
    tiles[..., 2048:] = scales.view(np.uint8).reshape(num_blocks, num_layers, 2, num_heads, 64)
    return torch.from_numpy(tiles).cuda()


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def assert_close(gpu: torch.Tensor, ref64: np.ndarray, what=""):
    g = to_f64(gpu)
    err = np.abs(g - ref64)
    bound = ATOL + RTOL * np.abs(ref64)
    bad = err > bound
    big = np.abs(ref64) >= 0.2
    max_rel = float((err[big] / np.abs(ref64[big])).max()) if big.any() else 0.0
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; "
                           f"max abs {err.max():.3g}, first at {np.argwhere(bad)[0]}")
    return float(err.max()), max_rel


def new_token_inputs(wl: workloads.Workload, layer: int, device="cuda"):
    """q, k_new, v_new for one layer of a workload, [T, H, 128] FP16."""
    T, H = wl.num_tokens, wl.num_heads
    q = workloads.normal_fp16((T, H, 128), workloads.value_seed(wl.seed, "q", layer)).to(device)
    k = workloads.normal_fp16((T, H, 128), workloads.value_seed(wl.seed, "k", layer)).to(device)
    v = workloads.normal_fp16((T, H, 128), workloads.value_seed(wl.seed, "v", layer)).to(device)
    return q, k, v


def step_metadata(wl: workloads.Workload, device="cuda"):
    """Device tables/ctx/q_start and the slots of the new tokens (oracle's slot function)."""
    slots = oracle.slots(wl.block_tables, wl.request_of_token(), wl.positions())
    return (torch.from_numpy(wl.block_tables).to(device), torch.from_numpy(wl.ctx_lens).to(device),
            torch.from_numpy(wl.q_start_loc()).to(device), torch.from_numpy(slots).to(device), slots)


def mini_pool(pool: torch.Tensor, layer: int, table_row: np.ndarray, nblocks: int):
    """Host copy of one layer of the blocks a row references, as a 1-layer pool
    with blocks renumbered 0..n-1 (a physical-block permutation, which the
    oracle's pins show leaves attention unchanged)."""
    ids = torch.from_numpy(table_row[:nblocks].astype(np.int64)).to(pool.device)
    sub = pool.index_select(0, ids)[:, layer:layer + 1].contiguous()
    return to_bits(sub).reshape(sub.shape), np.arange(nblocks, dtype=np.int32)
