"""The oracle: a plain CPU statement of what the paged KV cache path computes.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py`` call it; the library under
``paged_kv_cache_scatter_gb300`` never imports, links or runs anything here.
It shares no code with the CUDA path.

Every function follows a passage of the source pages (see the C file's
header for the page and section of each): the block layout and byte ledger,
the slot of a logical position, the append of a token's K/V, the gather of a
sequence's blocks into contiguous K and V, and softmax attention in double
precision, rounded to FP16 once at the end. ``blockmgr`` restates the
ref-counted block manager.

Pins (tests/test_oracle_pins.py): the pages' byte and block arithmetic, the
exhaustive binary16 table, a one-hot softmax whose output is exactly one V
row, the uniform-softmax mean, invariance under a permutation of physical
blocks, brute force against a float64 library attention on tiny inputs,
chunked prefill against unchunked causal attention, the split-merge
identity, and for grouped-query heads (GQA, MQA) a float64 library attention
with the K/V heads repeated plus the equality with an MHA pool whose head
groups hold identical K/V. The 8-bit cache (INT8 codes, one float32 scale per
(token, head) row) is pinned by the pages' halving of the cache bytes, exact
round trips of rows built from integer codes and power-of-two scales, the
half-step error bound and nearest-code rule checked in float64, byte
placement checked with numpy's own indexing, and attention over exactly
stored values equal to the FP16 pool's. Block copies and swaps are checked
byte for byte against numpy indexing; the chained prefix hash against the
published FNV-1a test vectors, its dependence on the whole prefix, and the
page's own cache lookup restated; the block manager's fork, copy-on-write,
swap and prefix cache against worked scenarios and reference-count
invariants under random operations. Parity is pinned for every function;
none is unpinned.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


class Geom(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("num_layers", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("dtype", ctypes.c_int32)]


FP16, INT8 = 0, 1


def lib():
    global _lib
    if _lib is None:
        # a test may point this at a deliberately broken copy (tests/test_oracle_mutants.py)
        path = os.environ.get("PKV_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        G = ctypes.POINTER(Geom)
        sig = {
            "pkvo_half_to_double": (dbl, [ctypes.c_uint16]),
            "pkvo_double_to_half": (ctypes.c_uint16, [dbl]),
            "pkvo_halves_to_doubles": (None, [P, P, i64]),
            "pkvo_doubles_to_halves": (None, [P, P, i64]),
            "pkvo_bytes_per_token": (i64, [G]),
            "pkvo_bytes_per_block": (i64, [G]),
            "pkvo_pool_bytes": (i64, [G]),
            "pkvo_blocks_for_tokens": (i64, [i64, i32]),
            "pkvo_slot": (i64, [P, i64, i32]),
            "pkvo_slots": (None, [P, i32, P, P, i64, i32, P]),
            "pkvo_kv_append": (i64, [P, G, ctypes.c_int, P, P, P, i64]),
            "pkvo_gather": (None, [P, G, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, i64, P]),
            "pkvo_attend": (None, [P, P, P, i64, ctypes.c_int, dbl, P]),
            "pkvo_decode_attn": (None, [P, G, ctypes.c_int, P, P, i32, P, i32, dbl, P, P]),
            "pkvo_prefill_attn": (None, [P, G, ctypes.c_int, P, P, P, i32, P, i32, dbl, P, P]),
            "pkvo_partial": (None, [P, P, P, i64, i64, ctypes.c_int, dbl, P, P, P]),
            "pkvo_merge": (None, [P, P, P, ctypes.c_int, ctypes.c_int, P]),
            "pkvo_decode_attn_split": (None, [P, G, ctypes.c_int, P, P, i32, P, i32, dbl, i64, P]),
            "pkvo_i8_tile_bytes": (i64, [G]),
            "pkvo_i8_quantize_row": (None, [P, ctypes.c_int, P, P]),
            "pkvo_i8_dequant": (dbl, [ctypes.c_int8, ctypes.c_float]),
            "pkvo_copy_blocks": (i64, [P, G, P, i64]),
            "pkvo_swap_out": (i64, [P, G, P, i64, P]),
            "pkvo_swap_in": (i64, [P, G, P, i64, P]),
            "pkvo_fnv1a64": (ctypes.c_uint64, [P, i64]),
            "pkvo_block_hashes": (i64, [P, i64, i32, P]),
            "pkvo_num_threads": (ctypes.c_int, []),
            "pkvo_set_num_threads": (None, [ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def geom(num_blocks, num_layers, num_heads=32, head_dim=128, block_size=16, num_q_heads=None,
         dtype=FP16) -> Geom:
    """num_heads: K/V heads stored in the pool; num_q_heads: query heads (default num_heads). Query head h
    reads K/V head h // (num_q_heads // num_heads) (grouped-query attention; one K/V head for all is MQA).
    dtype FP16: the pool is uint16 (binary16 bits); INT8: the pool is bytes, each (block, layer, K/V, head)
    tile holding 16 x head_dim int8 codes followed by 16 float32 scales."""
    return Geom(int(num_blocks), int(num_layers), int(num_heads), int(head_dim), int(block_size),
                int(num_q_heads or num_heads), int(dtype))


def _qh(g: Geom) -> int:
    """Query heads of a geometry (K/V heads when it has no grouping)."""
    return g.num_q_heads or g.num_heads


# ---------------------------------------------------------------- binary16

def half_to_double(bits) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    lib().pkvo_halves_to_doubles(_p(bits), _p(out), bits.size)
    return out


def double_to_half(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().pkvo_doubles_to_halves(_p(x), _p(out), x.size)
    return out


# ---------------------------------------------------------------- geometry

def bytes_per_token(g: Geom) -> int:
    return lib().pkvo_bytes_per_token(ctypes.byref(g))


def bytes_per_block(g: Geom) -> int:
    return lib().pkvo_bytes_per_block(ctypes.byref(g))


def pool_bytes(g: Geom) -> int:
    return lib().pkvo_pool_bytes(ctypes.byref(g))


def i8_tile_bytes(g: Geom) -> int:
    return lib().pkvo_i8_tile_bytes(ctypes.byref(g))


def i8_quantize_row(x_bits):
    """(int8 codes, float32 scale) of one row of FP16 values (uint16 bits)."""
    x = _c(x_bits, np.uint16)
    codes = np.empty(x.shape[0], np.int8)
    scale = ctypes.c_float()
    lib().pkvo_i8_quantize_row(_p(x), x.shape[0], _p(codes), ctypes.byref(scale))
    return codes, np.float32(scale.value)


def i8_dequant(code: int, scale) -> float:
    return lib().pkvo_i8_dequant(int(code), float(scale))


def empty_pool(g: Geom) -> np.ndarray:
    """A zeroed host pool of the geometry's element type (uint16 for FP16, bytes for INT8)."""
    if g.dtype == INT8:
        return np.zeros(pool_bytes(g), np.uint8)
    return np.zeros(pool_bytes(g) // 2, np.uint16)


def blocks_for_tokens(tokens: int, block_size: int = 16) -> int:
    return lib().pkvo_blocks_for_tokens(int(tokens), int(block_size))


def slots(tables, row_of_token, positions, block_size=16) -> np.ndarray:
    tables = _c(tables, np.int32)
    row_of_token = _c(row_of_token, np.int32)
    positions = _c(positions, np.int64)
    out = np.empty(positions.shape[0], np.int64)
    lib().pkvo_slots(_p(tables), tables.shape[1], _p(row_of_token), _p(positions), positions.shape[0],
                     block_size, _p(out))
    return out


# ------------------------------------------------------------ the kernels

def kv_append(pool: np.ndarray, g: Geom, layer: int, k, v, slot_mapping) -> int:
    """In-place on ``pool`` (uint16 view of FP16, or bytes for an INT8 geometry). Returns -1 or the first
    bad token index. k and v are FP16 bits [T, num_heads, head_dim]; an INT8 pool stores them quantised."""
    assert pool.dtype == (np.uint8 if g.dtype == INT8 else np.uint16) and pool.flags.c_contiguous
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    s = _c(slot_mapping, np.int64)
    return lib().pkvo_kv_append(_p(pool), ctypes.byref(g), layer, _p(k), _p(v), _p(s), s.shape[0])


def gather(pool: np.ndarray, g: Geom, layer: int, kv: int, head: int, table, seq_len: int) -> np.ndarray:
    table = _c(table, np.int32)
    out = np.empty((seq_len, g.head_dim), np.float64)
    lib().pkvo_gather(_p(pool), ctypes.byref(g), layer, kv, head, _p(table), seq_len, _p(out))
    return out


def attend(q, K, V, scale: float) -> np.ndarray:
    q = _c(q, np.float64)
    K = _c(K, np.float64)
    V = _c(V, np.float64)
    out = np.empty(q.shape[-1], np.float64)
    lib().pkvo_attend(_p(q), _p(K), _p(V), K.shape[0], q.shape[-1], float(scale), _p(out))
    return out


def decode_attn(pool, g: Geom, layer, q, tables, ctx_lens, scale, want_f16=True):
    """Returns (out_f64, out_f16_bits) with layout [B, heads, dim]."""
    q = _c(q, np.uint16)
    tables = _c(tables, np.int32)
    ctx = _c(ctx_lens, np.int32)
    B = ctx.shape[0]
    o64 = np.empty((B, _qh(g), g.head_dim), np.float64)
    o16 = np.empty((B, _qh(g), g.head_dim), np.uint16)
    lib().pkvo_decode_attn(_p(pool), ctypes.byref(g), layer, _p(q), _p(tables), tables.shape[1], _p(ctx), B,
                           float(scale), _p(o64), _p(o16))
    return o64, o16


def prefill_attn(pool, g: Geom, layer, q, q_start, tables, ctx_lens, scale):
    """Returns (out_f64, out_f16_bits) with layout [T, heads, dim]."""
    q = _c(q, np.uint16)
    qs = _c(q_start, np.int32)
    tables = _c(tables, np.int32)
    ctx = _c(ctx_lens, np.int32)
    S = ctx.shape[0]
    T = int(qs[-1])
    o64 = np.zeros((T, _qh(g), g.head_dim), np.float64)
    o16 = np.zeros((T, _qh(g), g.head_dim), np.uint16)
    lib().pkvo_prefill_attn(_p(pool), ctypes.byref(g), layer, _p(q), _p(qs), _p(tables), tables.shape[1],
                            _p(ctx), S, float(scale), _p(o64), _p(o16))
    return o64, o16


def partial(q, K, V, lo, hi, scale):
    q = _c(q, np.float64)
    K = _c(K, np.float64)
    V = _c(V, np.float64)
    m = ctypes.c_double()
    l = ctypes.c_double()
    o = np.empty(q.shape[-1], np.float64)
    lib().pkvo_partial(_p(q), _p(K), _p(V), lo, hi, q.shape[-1], float(scale), ctypes.byref(m), ctypes.byref(l),
                       _p(o))
    return m.value, l.value, o


def merge(m, l, o) -> np.ndarray:
    m = _c(m, np.float64)
    l = _c(l, np.float64)
    o = _c(o, np.float64)
    out = np.empty(o.shape[-1], np.float64)
    lib().pkvo_merge(_p(m), _p(l), _p(o), m.shape[0], o.shape[-1], _p(out))
    return out


def decode_attn_split(pool, g: Geom, layer, q, tables, ctx_lens, scale, part_tokens) -> np.ndarray:
    q = _c(q, np.uint16)
    tables = _c(tables, np.int32)
    ctx = _c(ctx_lens, np.int32)
    B = ctx.shape[0]
    o64 = np.empty((B, _qh(g), g.head_dim), np.float64)
    lib().pkvo_decode_attn_split(_p(pool), ctypes.byref(g), layer, _p(q), _p(tables), tables.shape[1], _p(ctx), B,
                                 float(scale), int(part_tokens), _p(o64))
    return o64


# ------------------------------------------------------------ block copy, swap, prefix hashes

def copy_blocks(pool: np.ndarray, g: Geom, pairs) -> int:
    """In place: block dst receives block src for each (src, dst) row of ``pairs``. -1 or the first bad pair."""
    pr = _c(pairs, np.int32).reshape(-1, 2)
    return lib().pkvo_copy_blocks(_p(pool), ctypes.byref(g), _p(pr), pr.shape[0])


def swap_out(pool: np.ndarray, g: Geom, blocks) -> np.ndarray:
    """The listed whole blocks, concatenated (bytes), as swap-out writes them to host memory."""
    b = _c(blocks, np.int32)
    out = np.empty(b.shape[0] * bytes_per_block(g), np.uint8)
    r = lib().pkvo_swap_out(_p(pool), ctypes.byref(g), _p(b), b.shape[0], _p(out))
    if r != -1:
        raise IndexError(f"block index {r} outside the pool")
    return out


def swap_in(pool: np.ndarray, g: Geom, blocks, host_bytes) -> int:
    b = _c(blocks, np.int32)
    h = _c(host_bytes, np.uint8)
    return lib().pkvo_swap_in(_p(pool), ctypes.byref(g), _p(b), b.shape[0], _p(h))


def fnv1a64(data: bytes) -> int:
    buf = np.frombuffer(bytes(data), np.uint8).copy() if len(data) else np.zeros(1, np.uint8)
    return int(lib().pkvo_fnv1a64(_p(buf), len(data)))


def block_hashes(tokens, block_size: int = 16) -> np.ndarray:
    """Chained hashes of the full blocks of a token-id stream (uint64)."""
    t = _c(tokens, np.int32)
    out = np.zeros(max(1, t.shape[0] // block_size), np.uint64)
    n = lib().pkvo_block_hashes(_p(t), t.shape[0], block_size, _p(out))
    return out[:n]


def num_threads() -> int:
    return lib().pkvo_num_threads()


def set_num_threads(n: int) -> None:
    lib().pkvo_set_num_threads(int(n))


SCALE_FP32 = float(np.float32(1.0 / np.sqrt(np.float32(128.0))))
