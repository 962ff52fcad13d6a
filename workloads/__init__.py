"""Seeded synthetic inputs for the paged KV cache path.

This module draws random numbers and lays block ids out from a random
permutation; it holds none of the scatter or attention arithmetic. The
oracle tests, the CUDA parity tests and ``bench.py`` all take their inputs
from here, so both sides of every comparison see the same bytes.

The shapes follow the design problem on the page "llm-inference-batching"
(faangrind), sections "Model" and "KV cache": a 7B model with 32 layers,
32 heads, head dimension 128, FP16, and a pool of 7,152 blocks of 16 tokens.
The length mix follows the same page's opening paragraph (prompts of 50 to
8,000 tokens, answers up to 1,000) and "How many requests fit" (an average
request of 1,250 prompt tokens).

Recipe (seed 0 unless stated):
  * lengths and block permutations: ``numpy.random.default_rng(seed)``;
  * block ids: ``rng.permutation(num_blocks)`` handed out in row order, each
    row taking ceil(ctx / 16) consecutive entries of the permutation;
  * values: N(0, 1) drawn in FP32 by ``torch.Generator`` and cast to FP16
    (round to nearest even).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

NUM_LAYERS = 32
NUM_HEADS = 32
HEAD_DIM = 128
BLOCK_SIZE = 16
POOL_BLOCKS = 7152          # 60 GB pool / 8,388,608 B per block
PREFILL_CHUNK = 512


@dataclass
class Workload:
    """One engine iteration's metadata: rows, their contexts and new tokens.

    Rows with ``q_lens == 1`` are decode rows and come first; rows with
    ``q_lens > 1`` are prefill chunks. ``ctx_lens`` counts the cached tokens a
    row attends, including the ones appended in this iteration.
    """
    name: str
    num_layers: int
    num_blocks: int
    block_tables: np.ndarray     # int32 [S, max_blocks], -1 where unused
    ctx_lens: np.ndarray         # int32 [S]
    q_lens: np.ndarray           # int32 [S]
    seed: int
    num_heads: int = NUM_HEADS   # K/V heads stored in the pool
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    meta: dict = field(default_factory=dict)
    num_q_heads: int = 0         # query heads; 0 = num_heads (grouped-query attention when larger)

    @property
    def q_heads(self) -> int:
        return self.num_q_heads or self.num_heads

    @property
    def num_seqs(self) -> int:
        return int(self.ctx_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_tokens(self) -> int:
        return int(self.q_lens.sum())

    @property
    def num_decode(self) -> int:
        return int((self.q_lens == 1).sum())

    def q_start_loc(self) -> np.ndarray:
        out = np.zeros(self.num_seqs + 1, dtype=np.int32)
        out[1:] = np.cumsum(self.q_lens)
        return out

    def positions(self) -> np.ndarray:
        """Logical position of each new token, in flat token order."""
        pos = [np.arange(c - q, c, dtype=np.int64) for c, q in zip(self.ctx_lens, self.q_lens)]
        return np.concatenate(pos) if pos else np.zeros(0, np.int64)

    def request_of_token(self) -> np.ndarray:
        return np.repeat(np.arange(self.num_seqs, dtype=np.int32), self.q_lens)


def _tables_from_perm(perm: np.ndarray, nblocks_per_row, shared: np.ndarray | None = None) -> np.ndarray:
    """Hand out block ids from ``perm`` in row order (after an optional shared prefix)."""
    nshared = 0 if shared is None else len(shared)
    width = max(nshared + int(n) for n in nblocks_per_row) if len(nblocks_per_row) else 1
    tables = np.full((len(nblocks_per_row), width), -1, dtype=np.int32)
    cursor = 0
    for r, n in enumerate(nblocks_per_row):
        if nshared:
            tables[r, :nshared] = shared
        tables[r, nshared:nshared + n] = perm[cursor:cursor + n]
        cursor += int(n)
    if cursor > len(perm):
        raise ValueError("workload needs more blocks than the pool holds")
    return tables


def _blocks_for(n: int, bs: int = BLOCK_SIZE) -> int:
    return -(-int(n) // bs)


# ---------------------------------------------------------------------------
# length draws

def clipped_lognormal_mean(mu: float, sigma: float, lo: float, hi: float) -> float:
    """Mean of min(max(X, lo), hi) for X ~ LogNormal(mu, sigma), in closed form."""
    def phi(z):
        return 0.5 * (1.0 + math.erf(z / math.sqrt(2.0)))
    a, b = math.log(lo), math.log(hi)
    below = phi((a - mu) / sigma)
    above = 1.0 - phi((b - mu) / sigma)
    inside = math.exp(mu + sigma * sigma / 2) * (phi((b - mu - sigma * sigma) / sigma)
                                                  - phi((a - mu - sigma * sigma) / sigma))
    return lo * below + hi * above + inside


def lognormal_mu_for_mean(mean: float, sigma: float, lo: float, hi: float) -> float:
    """Bisect mu so that the clipped distribution has the requested mean."""
    a, b = math.log(lo), math.log(hi)
    for _ in range(200):
        m = 0.5 * (a + b)
        if clipped_lognormal_mean(m, sigma, lo, hi) < mean:
            a = m
        else:
            b = m
    return 0.5 * (a + b)


# ---------------------------------------------------------------------------
# the five workloads

def tiny_decode(seed: int = 0) -> Workload:
    """1 layer, 4 rows, contexts 17/50/100/255, 64-block permuted pool."""
    rng = np.random.default_rng(seed)
    ctx = np.array([17, 50, 100, 255], dtype=np.int32)
    perm = rng.permutation(64).astype(np.int32)
    tables = _tables_from_perm(perm, [_blocks_for(c) for c in ctx])
    return Workload("tiny_decode", 1, 64, tables, ctx, np.ones(4, np.int32), seed)


def average_decode(seed: int = 0, num_layers: int = NUM_LAYERS, num_blocks: int = POOL_BLOCKS,
                   batch: int = 32) -> Workload:
    """Batch-32 decode: prompt ~ clipped lognormal (mean 1,250) + generated U{0..299} + 1."""
    rng = np.random.default_rng(seed)
    mu = lognormal_mu_for_mean(1250.0, 1.0, 50.0, 8000.0)
    prompt = np.rint(np.clip(rng.lognormal(mu, 1.0, batch), 50, 8000)).astype(np.int64)
    generated = rng.integers(0, 300, batch)
    ctx = (prompt + generated + 1).astype(np.int32)
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = _tables_from_perm(perm, [_blocks_for(c) for c in ctx])
    return Workload("average_decode", num_layers, num_blocks, tables, ctx, np.ones(batch, np.int32), seed,
                    meta={"mu": mu, "sigma": 1.0, "prompt": prompt.tolist(), "generated": generated.tolist()})


def long_decode(seed: int = 0, num_layers: int = NUM_LAYERS, num_blocks: int = POOL_BLOCKS,
                batch: int = 13, ctx_len: int = 8192) -> Workload:
    """13 rows at 8,192 context tokens each (512 blocks per row)."""
    rng = np.random.default_rng(seed)
    ctx = np.full(batch, ctx_len, dtype=np.int32)
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = _tables_from_perm(perm, [_blocks_for(c) for c in ctx])
    return Workload("long_decode", num_layers, num_blocks, tables, ctx, np.ones(batch, np.int32), seed)


def mixed_prefill(chunk: int, seed: int = 0, num_layers: int = NUM_LAYERS, num_blocks: int = POOL_BLOCKS,
                  prompt_len: int = 4000, decode_rows: int = 31, chunk_size: int = PREFILL_CHUNK) -> Workload:
    """Chunk ``chunk`` of a ``prompt_len`` prompt plus ``decode_rows`` decode rows.

    Chunk i covers prompt positions [chunk_size*i, min(chunk_size*(i+1), prompt_len)).
    Decode rows start at a context drawn from U{100..2000} and advance one
    token per chunk iteration. Block tables are laid out for the final length,
    so they are the same for every chunk of the schedule.
    """
    nchunks = -(-prompt_len // chunk_size)
    if not 0 <= chunk < nchunks:
        raise ValueError("chunk out of range")
    rng = np.random.default_rng(seed)
    base = rng.integers(100, 2001, decode_rows).astype(np.int64)
    final = base + (nchunks - 1)
    perm = rng.permutation(num_blocks).astype(np.int32)
    nblk = [_blocks_for(c) for c in final] + [_blocks_for(prompt_len)]
    tables = _tables_from_perm(perm, nblk)
    start = chunk_size * chunk
    end = min(start + chunk_size, prompt_len)
    ctx = np.concatenate([base + chunk, [end]]).astype(np.int32)
    qlen = np.concatenate([np.ones(decode_rows, np.int64), [end - start]]).astype(np.int32)
    return Workload(f"mixed_prefill_chunk{chunk}", num_layers, num_blocks, tables, ctx, qlen, seed,
                    meta={"chunk": chunk, "chunk_start": start, "chunk_end": end, "prompt_len": prompt_len,
                          "num_chunks": nchunks})


def shared_prefix_decode(seed: int = 0, num_layers: int = NUM_LAYERS, num_blocks: int = POOL_BLOCKS,
                         batch: int = 64, prefix_blocks: int = 125) -> Workload:
    """64 rows sharing 125 full prefix blocks, then 1..300 private tokens each."""
    rng = np.random.default_rng(seed)
    u = rng.integers(1, 301, batch)
    ctx = (prefix_blocks * BLOCK_SIZE + u).astype(np.int32)
    perm = rng.permutation(num_blocks).astype(np.int32)
    shared = perm[:prefix_blocks]
    tables = _tables_from_perm(perm[prefix_blocks:], [_blocks_for(x) for x in u], shared=shared)
    return Workload("shared_prefix_decode", num_layers, num_blocks, tables, ctx, np.ones(batch, np.int32), seed,
                    meta={"prefix_blocks": prefix_blocks, "private_tokens": u.tolist()})


GQA_KV_HEADS = 8
GQA_POOL_BLOCKS = 28608     # 60 GB / 2,097,152 B per block (8 K/V heads, 32 layers)


def gqa_decode(seed: int = 0, num_layers: int = NUM_LAYERS, num_blocks: int = GQA_POOL_BLOCKS,
               batch: int = 32, ctx_len: int = 2300, kv_heads: int = GQA_KV_HEADS,
               q_heads: int = NUM_HEADS) -> Workload:
    """Grouped-query decode: 32 rows at 2,300 context tokens, 8 K/V heads serving 32 query heads
    (131,072 B of K/V per token over 32 layers, so one step reads 9.65 GB), shuffled 60 GB pool."""
    rng = np.random.default_rng(seed)
    ctx = np.full(batch, ctx_len, dtype=np.int32)
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = _tables_from_perm(perm, [_blocks_for(c) for c in ctx])
    return Workload("gqa_decode", num_layers, num_blocks, tables, ctx, np.ones(batch, np.int32), seed,
                    num_heads=kv_heads, num_q_heads=q_heads)


def random_step(seed: int, num_seqs: int, max_ctx: int, num_blocks: int, num_layers: int = 1,
                prefill_rows: int = 0, max_q: int = 64, min_ctx: int = 1) -> Workload:
    """Small random ragged step for parity tests: decode rows, then prefill rows."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(min_ctx, max_ctx + 1, num_seqs).astype(np.int32)
    qlen = np.ones(num_seqs, np.int32)
    for r in range(num_seqs - prefill_rows, num_seqs):
        qlen[r] = int(rng.integers(2, max(3, min(max_q, int(ctx[r])) + 1))) if ctx[r] >= 2 else 1
        qlen[r] = min(qlen[r], ctx[r])
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = _tables_from_perm(perm, [_blocks_for(c) for c in ctx])
    return Workload(f"random_step_{seed}", num_layers, num_blocks, tables, ctx, qlen, seed)


# ---------------------------------------------------------------------------
# values

def value_seed(seed: int, tag: str, layer: int = 0) -> int:
    tags = {"pool": 1, "q": 2, "k": 3, "v": 4}
    return (seed * 1_000_003 + tags[tag] * 10_007 + layer) & 0x7FFFFFFF


def normal_fp16(shape, seed: int, device="cpu"):
    """N(0,1) drawn in FP32 by a seeded torch generator, rounded to FP16."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.float16)


def fill_normal_fp16_(t, seed: int, chunk_elems: int = 1 << 28):
    """Fill a (possibly huge) FP16 tensor in place with N(0,1), chunk by chunk."""
    import torch
    gen = torch.Generator(device=t.device)
    gen.manual_seed(seed)
    flat = t.view(-1)
    tmp = None
    for s in range(0, flat.numel(), chunk_elems):
        n = min(chunk_elems, flat.numel() - s)
        if tmp is None or tmp.numel() < n:
            tmp = torch.empty(n, dtype=torch.float32, device=t.device)
        tmp[:n].normal_(generator=gen)
        flat[s:s + n].copy_(tmp[:n])
    return t


def fill_int8_tiles_(t, seed: int, scale: float = 0.02, chunk_tiles: int = 1 << 17):
    """Fill an 8-bit pool (uint8 tensor of whole 2,112-byte tiles) in place: codes uniform in [-127, 127],
    every scale ``scale`` (about what N(0,1) rows quantise to), chunk by chunk on the tensor's device."""
    import torch
    tiles = t.view(-1, 2112)
    gen = torch.Generator(device=t.device)
    gen.manual_seed(seed)
    sbytes = torch.full((16,), scale, dtype=torch.float32).view(torch.uint8).to(t.device)
    for s in range(0, tiles.shape[0], chunk_tiles):
        n = min(chunk_tiles, tiles.shape[0] - s)
        codes = torch.randint(-127, 128, (n, 2048), generator=gen, device=t.device, dtype=torch.int16)
        tiles[s:s + n, :2048].copy_(codes.to(torch.int8).view(torch.uint8))
        tiles[s:s + n, 2048:].copy_(sbytes.expand(n, 64))
    return t


def pool_shape(num_blocks: int, num_layers: int, num_heads: int = NUM_HEADS, head_dim: int = HEAD_DIM,
               block_size: int = BLOCK_SIZE):
    """[block, layer, K/V, head, token-in-block, dim] — one block holds every layer."""
    return (num_blocks, num_layers, 2, num_heads, block_size, head_dim)
