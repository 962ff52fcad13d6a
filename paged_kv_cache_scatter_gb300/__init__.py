"""Paged KV cache kernels for GB300 (sm_103a): Python binding of libpkv.

Argument marshalling only — every step of the path runs in libpkv's CUDA
kernels. The raw C entry points are exposed under their C names
(``pkv_kv_append``, ``pkv_decode_attn``, ...); ``Pool`` wraps a pool handle
and accepts torch tensors, passing their device pointers and the current
CUDA stream. If ``libpkv.so`` has not been built the import fails loudly:
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpkv.so")

PKV_OK, PKV_E_INVALID, PKV_E_NOMEM, PKV_E_SHARED, PKV_E_DEVICE, PKV_E_TIMEOUT = range(6)
PKV_DEV_BAD_SLOT, PKV_DEV_BAD_BLOCK, PKV_DEV_BAD_CTX, PKV_DEV_BAD_QLEN, PKV_DEV_TIMEOUT = 1, 2, 4, 8, 16
PKV_DTYPE_FP16 = 0
PKV_DTYPE_INT8 = 1
_DTYPES = {"fp16": PKV_DTYPE_FP16, "int8": PKV_DTYPE_INT8}

_c = ctypes
_P = _c.c_void_p
_i32, _i64, _u32, _u64, _f32, _sz = _c.c_int32, _c.c_int64, _c.c_uint32, _c.c_uint64, _c.c_float, _c.c_size_t


class pkv_pool_desc(_c.Structure):
    _fields_ = [("num_blocks", _i64), ("num_layers", _i32), ("num_heads", _i32), ("head_dim", _i32),
                ("block_size", _i32), ("dtype", _i32), ("partition_tokens", _i32), ("dev_base", _P),
                ("bytes", _sz), ("free_order", _P), ("num_q_heads", _i32)]


class pkv_step_desc(_c.Structure):
    _fields_ = [("num_decode", _i32), ("num_prefill", _i32), ("num_tokens", _i32), ("max_q_len", _i32),
                ("max_blocks", _i32), ("first_layer", _i32), ("num_layers", _i32), ("scale", _f32),
                ("block_tables", _P), ("ctx_lens", _P), ("q_start_loc", _P), ("slot_mapping", _P),
                ("q", _P), ("k", _P), ("v", _P), ("out", _P),
                ("q_layer_stride", _i64), ("k_layer_stride", _i64), ("v_layer_stride", _i64),
                ("out_layer_stride", _i64)]


_PD = _c.POINTER(pkv_pool_desc)
_SD = _c.POINTER(pkv_step_desc)

# name -> (restype, argtypes); the C declarations are in include/pkv.h
SIGNATURES = {
    "pkv_pool_bytes": (_sz, [_PD]),
    "pkv_pool_create": (_i32, [_PD, _c.POINTER(_P)]),
    "pkv_pool_destroy": (_i32, [_P]),
    "pkv_seq_grow": (_i32, [_P, _i64, _i64]),
    "pkv_seq_share_prefix": (_i32, [_P, _i64, _i64, _i64]),
    "pkv_seq_free": (_i32, [_P, _i64]),
    "pkv_free_blocks": (_i64, [_P]),
    "pkv_ref_count": (_i32, [_P, _i64]),
    "pkv_seq_len": (_i64, [_P, _i64]),
    "pkv_block_table": (_i32, [_P, _i64, _P, _i64, _c.POINTER(_i64)]),
    "pkv_seq_fork": (_i32, [_P, _i64, _i64]),
    "pkv_seq_cow": (_i32, [_P, _i64, _i64, _c.POINTER(_i32), _c.POINTER(_i32)]),
    "pkv_seq_swap_out": (_i32, [_P, _i64, _P, _i64, _c.POINTER(_i64)]),
    "pkv_seq_swap_in": (_i32, [_P, _i64, _P, _i64, _c.POINTER(_i64)]),
    "pkv_block_hashes": (_i64, [_P, _i64, _P, _i64]),
    "pkv_prefix_register": (_i32, [_P, _i64, _P, _i64, _c.POINTER(_i64)]),
    "pkv_prefix_match": (_i64, [_P, _P, _i64]),
    "pkv_seq_attach_prefix": (_i32, [_P, _i64, _P, _i64, _c.POINTER(_i64)]),
    "pkv_prefix_evict": (_i64, [_P, _i64]),
    "pkv_prefix_cached_blocks": (_i64, [_P]),
    "pkv_copy_blocks": (_i32, [_P, _P, _i32, _P]),
    "pkv_swap_blocks_out": (_i32, [_P, _P, _i32, _P, _P]),
    "pkv_swap_blocks_in": (_i32, [_P, _P, _i32, _P, _P]),
    "pkv_build_step": (_i32, [_P, _P, _P, _i32, _i32, _P, _P, _P, _P]),
    "pkv_kv_append": (_i32, [_P, _i32, _P, _P, _P, _i32, _P]),
    "pkv_decode_workspace_bytes": (_sz, [_P, _i32, _i32]),
    "pkv_decode_attn": (_i32, [_P, _i32, _P, _P, _i32, _P, _i32, _f32, _P, _P, _sz, _P]),
    "pkv_prefill_attn": (_i32, [_P, _i32, _P, _P, _P, _i32, _P, _i32, _i32, _f32, _P, _P]),
    "pkv_decode_attn_noalloc": (_i32, [_P, _i32, _P, _P, _i32, _P, _i32, _f32, _P, _P]),
    "pkv_decode_attn_cascade": (_i32, [_P, _i32, _P, _P, _i32, _P, _i32, _P, _P, _i32, _i32, _f32, _P, _P, _sz, _P]),
    "pkv_decode_cascade_workspace_bytes": (_sz, [_P, _i32, _i32]),
    "pkv_cascade_groups": (_i32, [_P, _P, _i32, _i32, _i32, _P, _P, _c.POINTER(_i32), _c.POINTER(_i32)]),
    "pkv_step_workspace_bytes": (_sz, [_P, _SD]),
    "pkv_step": (_i32, [_P, _SD, _P, _sz, _P]),
    "pkv_get_status": (_i32, [_P, _P, _c.POINTER(_u32)]),
    "pkv_last_error_string": (_c.c_char_p, []),
    "pkv_status_string": (_c.c_char_p, [_i32]),
    "pkv_debug_wait_probe": (_i32, [_P, _u64, _P]),
}

_lib = None


def load():
    """Load libpkv.so (built by ``paged_kv_cache_scatter_gb300.build``). No fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpkv.so is not built ({LIB_PATH}); run `python -m paged_kv_cache_scatter_gb300.build`")
        lib = _c.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
            globals()[name] = fn
        _lib = lib
    return _lib


class PkvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


def _check(status: int) -> None:
    if status != PKV_OK:
        raise PkvError(status, load().pkv_last_error_string().decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Pool:
    """A pool handle bound to a caller-owned device allocation (a torch tensor).

    With ``storage=None`` the handle is a host-only block manager: its
    bookkeeping calls work without a GPU and its kernel calls are refused."""

    def __init__(self, storage, num_blocks: int, num_layers: int = 32, num_heads: int = 32,
                 partition_tokens: int = 0, free_order=None, num_q_heads: int = 0, dtype: str = "fp16"):
        """num_heads: K/V heads stored per layer; num_q_heads: query heads (0 = num_heads), a multiple
        of num_heads (grouped-query attention: query head h reads K/V head h // (num_q_heads // num_heads)).
        dtype "fp16" or "int8" (the 8-bit cache: 2,112-byte tiles of INT8 codes and FP32 scales; the
        storage is then any device buffer of pkv_pool_bytes bytes, e.g. a uint8 tensor)."""
        lib = load()
        self._storage = storage
        self.num_blocks, self.num_layers, self.num_heads = int(num_blocks), int(num_layers), int(num_heads)
        self.num_q_heads = int(num_q_heads) or self.num_heads
        self.dtype = dtype
        self._order = None
        if free_order is not None:
            import numpy as np
            self._order = np.ascontiguousarray(free_order, dtype=np.int64)
        self.desc = pkv_pool_desc(self.num_blocks, self.num_layers, self.num_heads, 128, 16, _DTYPES[dtype],
                                  int(partition_tokens), _ptr(storage),
                                  0 if storage is None else storage.numel() * storage.element_size(),
                                  None if self._order is None else self._order.ctypes.data, self.num_q_heads)
        h = _P()
        _check(lib.pkv_pool_create(_c.byref(self.desc), _c.byref(h)))
        self.handle = h

    @staticmethod
    def bytes_needed(num_blocks: int, num_layers: int = 32, num_heads: int = 32, dtype: str = "fp16") -> int:
        d = pkv_pool_desc(int(num_blocks), int(num_layers), int(num_heads), 128, 16, _DTYPES[dtype], 0, None, 0, None)
        return load().pkv_pool_bytes(_c.byref(d))

    def close(self):
        if getattr(self, "handle", None):
            load().pkv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- block manager (host)
    def seq_grow(self, seq_id: int, new_len: int) -> int:
        return load().pkv_seq_grow(self.handle, seq_id, new_len)

    def seq_share_prefix(self, dst: int, src: int, n_blocks: int) -> int:
        return load().pkv_seq_share_prefix(self.handle, dst, src, n_blocks)

    def seq_free(self, seq_id: int) -> int:
        return load().pkv_seq_free(self.handle, seq_id)

    def free_blocks(self) -> int:
        return load().pkv_free_blocks(self.handle)

    def ref_count(self, block: int) -> int:
        return load().pkv_ref_count(self.handle, block)

    def seq_len(self, seq_id: int) -> int:
        return load().pkv_seq_len(self.handle, seq_id)

    def block_table(self, seq_id: int):
        import numpy as np
        n = _i64()
        st = load().pkv_block_table(self.handle, seq_id, None, 0, _c.byref(n))
        out = np.empty(max(n.value, 1), np.int32)
        _check(load().pkv_block_table(self.handle, seq_id, out.ctypes.data, out.shape[0], _c.byref(n)))
        return out[:n.value]

    def build_step(self, seq_ids, q_lens, max_blocks: int):
        """Returns (status, block_tables, ctx_lens, slot_mapping, q_start_loc) as numpy arrays."""
        import numpy as np
        sid = np.ascontiguousarray(seq_ids, np.int64)
        ql = np.ascontiguousarray(q_lens, np.int32)
        S = sid.shape[0]
        tables = np.empty((S, max_blocks), np.int32)
        ctx = np.empty(S, np.int32)
        slots = np.empty(max(int(ql.sum()), 1), np.int64)
        qs = np.empty(S + 1, np.int32)
        st = load().pkv_build_step(self.handle, sid.ctypes.data, ql.ctypes.data, S, max_blocks, tables.ctypes.data,
                                   ctx.ctypes.data, slots.ctypes.data, qs.ctypes.data)
        return st, tables, ctx, slots[:int(ql.sum())], qs

    # ---- copy-on-write, swap, prefix cache (host bookkeeping)
    def seq_fork(self, dst: int, src: int) -> int:
        return load().pkv_seq_fork(self.handle, dst, src)

    def seq_cow(self, seq_id: int, num_new: int = 1):
        """(status, src_block, dst_block) before a step writes the last num_new positions; (OK, -1, -1)
        when no copy is needed."""
        a, b = _i32(), _i32()
        st = load().pkv_seq_cow(self.handle, seq_id, num_new, _c.byref(a), _c.byref(b))
        return st, a.value, b.value

    def _swap(self, fn, seq_id: int):
        import numpy as np
        n = _i64()
        length = max(self.seq_len(seq_id), 0)
        out = np.empty(max((length + 15) // 16, 1), np.int32)   # a table never holds more blocks than this
        st = fn(self.handle, seq_id, out.ctypes.data, out.shape[0], _c.byref(n))
        return st, out[:n.value] if st == PKV_OK else None

    def seq_swap_out(self, seq_id: int):
        """(status, blocks to copy to host, in table order); the blocks are released."""
        return self._swap(load().pkv_seq_swap_out, seq_id)

    def seq_swap_in(self, seq_id: int):
        """(status, fresh blocks for the host copy to return to)."""
        return self._swap(load().pkv_seq_swap_in, seq_id)

    def prefix_register(self, seq_id: int, hashes):
        import numpy as np
        h = np.ascontiguousarray(hashes, np.uint64)
        n = _i64()
        st = load().pkv_prefix_register(self.handle, seq_id, h.ctypes.data if h.size else None, h.shape[0],
                                        _c.byref(n))
        return st, n.value

    def prefix_match(self, hashes) -> int:
        import numpy as np
        h = np.ascontiguousarray(hashes, np.uint64)
        return load().pkv_prefix_match(self.handle, h.ctypes.data if h.size else None, h.shape[0])

    def seq_attach_prefix(self, seq_id: int, hashes):
        import numpy as np
        h = np.ascontiguousarray(hashes, np.uint64)
        n = _i64()
        st = load().pkv_seq_attach_prefix(self.handle, seq_id, h.ctypes.data if h.size else None, h.shape[0],
                                          _c.byref(n))
        return st, n.value

    def prefix_evict(self, max_blocks: int) -> int:
        return load().pkv_prefix_evict(self.handle, max_blocks)

    def prefix_cached_blocks(self) -> int:
        return load().pkv_prefix_cached_blocks(self.handle)

    # ---- kernels (device tensors)
    def copy_blocks(self, pairs, stream=None) -> None:
        """pairs: device int32 [n, 2] of (src, dst) blocks."""
        _check(load().pkv_copy_blocks(self.handle, _ptr(pairs), int(pairs.shape[0]), _stream(stream)))

    def swap_blocks_out(self, blocks, host, stream=None) -> None:
        """blocks: device int32 [n]; host: pinned tensor of n * block bytes."""
        _check(load().pkv_swap_blocks_out(self.handle, _ptr(blocks), int(blocks.shape[0]), _ptr(host),
                                          _stream(stream)))

    def swap_blocks_in(self, blocks, host, stream=None) -> None:
        _check(load().pkv_swap_blocks_in(self.handle, _ptr(blocks), int(blocks.shape[0]), _ptr(host),
                                         _stream(stream)))

    def kv_append(self, layer: int, k, v, slot_mapping, stream=None) -> None:
        _check(load().pkv_kv_append(self.handle, layer, _ptr(k), _ptr(v), _ptr(slot_mapping),
                                    int(slot_mapping.shape[0]), _stream(stream)))

    def decode_workspace_bytes(self, num_seqs: int, max_blocks: int) -> int:
        return load().pkv_decode_workspace_bytes(self.handle, num_seqs, max_blocks)

    def decode_attn(self, layer: int, q, block_tables, ctx_lens, scale: float, out, workspace=None,
                    stream=None) -> None:
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check(load().pkv_decode_attn(self.handle, layer, _ptr(q), _ptr(block_tables), int(block_tables.shape[1]),
                                      _ptr(ctx_lens), int(ctx_lens.shape[0]), float(scale), _ptr(out),
                                      _ptr(workspace), ws_bytes, _stream(stream)))

    def decode_attn_noalloc(self, layer: int, q, block_tables, ctx_lens, scale: float, out, stream=None) -> None:
        """pkv_decode_attn without a workspace: the library's built-in 16 MiB scratch is used."""
        _check(load().pkv_decode_attn_noalloc(self.handle, layer, _ptr(q), _ptr(block_tables),
                                              int(block_tables.shape[1]), _ptr(ctx_lens), int(ctx_lens.shape[0]),
                                              float(scale), _ptr(out), _stream(stream)))

    def decode_cascade_workspace_bytes(self, num_seqs: int, max_blocks: int) -> int:
        return load().pkv_decode_cascade_workspace_bytes(self.handle, num_seqs, max_blocks)

    def decode_attn_cascade(self, layer: int, q, block_tables, ctx_lens, groups, scale: float, out, workspace=None,
                            stream=None) -> None:
        """groups = (group_start device int32 [G+1], group_blocks device int32 [G], max_group_rows)."""
        gs, gb, widest = groups
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check(load().pkv_decode_attn_cascade(self.handle, layer, _ptr(q), _ptr(block_tables),
                                              int(block_tables.shape[1]), _ptr(ctx_lens), int(ctx_lens.shape[0]),
                                              _ptr(gs), _ptr(gb), int(gb.shape[0]), int(widest), float(scale),
                                              _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)))

    def prefill_attn(self, layer: int, q, q_start_loc, block_tables, ctx_lens, max_q_len: int, scale: float, out,
                     stream=None) -> None:
        _check(load().pkv_prefill_attn(self.handle, layer, _ptr(q), _ptr(q_start_loc), _ptr(block_tables),
                                       int(block_tables.shape[1]), _ptr(ctx_lens), int(ctx_lens.shape[0]),
                                       int(max_q_len), float(scale), _ptr(out), _stream(stream)))

    def step_workspace_bytes(self, step: pkv_step_desc) -> int:
        return load().pkv_step_workspace_bytes(self.handle, _c.byref(step))

    def step(self, step: pkv_step_desc, workspace=None, stream=None) -> None:
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check(load().pkv_step(self.handle, _c.byref(step), _ptr(workspace), ws_bytes, _stream(stream)))

    def get_status(self, stream=None):
        """(status, device_flags); syncs the stream and clears the device error word."""
        flags = _u32()
        st = load().pkv_get_status(self.handle, _stream(stream), _c.byref(flags))
        return st, flags.value

    def debug_wait_probe(self, timeout_ns: int, stream=None) -> None:
        _check(load().pkv_debug_wait_probe(self.handle, int(timeout_ns), _stream(stream)))


def cascade_groups(tables, ctx_lens, min_rows: int = 2):
    """(group_start int32 [G+1], group_blocks int32 [G], max_group_rows) from host tables / lengths."""
    import numpy as np
    t = np.ascontiguousarray(tables, np.int32)
    c = np.ascontiguousarray(ctx_lens, np.int32)
    B = t.shape[0]
    gs = np.zeros(B + 1, np.int32)
    gb = np.zeros(max(B, 1), np.int32)
    G, W = _i32(), _i32()
    _check(load().pkv_cascade_groups(t.ctypes.data, c.ctypes.data, B, t.shape[1], int(min_rows), gs.ctypes.data,
                                     gb.ctypes.data, _c.byref(G), _c.byref(W)))
    return gs[:G.value + 1], gb[:G.value], W.value


def block_hashes(tokens):
    """Chained prefix hashes (uint64) of the full blocks of a host int32 token-id array."""
    import numpy as np
    t = np.ascontiguousarray(tokens, np.int32)
    out = np.empty(max(1, t.shape[0] // 16), np.uint64)
    n = load().pkv_block_hashes(t.ctypes.data if t.size else None, t.shape[0], out.ctypes.data, out.shape[0])
    if n < 0:
        raise PkvError(PKV_E_INVALID, "bad token array")
    return out[:n]


def make_step_desc(*, num_decode, num_prefill, num_tokens, max_q_len, max_blocks, first_layer, num_layers, scale,
                   block_tables, ctx_lens, q_start_loc, slot_mapping, q, k, v, out,
                   q_layer_stride, k_layer_stride, v_layer_stride, out_layer_stride) -> pkv_step_desc:
    return pkv_step_desc(int(num_decode), int(num_prefill), int(num_tokens), int(max_q_len), int(max_blocks),
                         int(first_layer), int(num_layers), float(scale), _ptr(block_tables), _ptr(ctx_lens),
                         _ptr(q_start_loc), _ptr(slot_mapping), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                         int(q_layer_stride), int(k_layer_stride), int(v_layer_stride), int(out_layer_stride))
