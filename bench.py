"""Benchmark: one engine iteration (32 layers) of the paged KV cache path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one pass of the whole hot path over one batch, through libpkv's C
ABI (pkv_step): for each of the 32 layers, kv_append of every new token,
decode attention of every decode row over its paged context, and causal
prefill attention of every prompt chunk. Default workload (the headline):
batch-32 decode with prompt lengths from a clipped lognormal (mean 1,250,
50..8,000) plus U{0..299} generated tokens, over a 7,152-block (60 GB) pool
with shuffled block ids, N(0,1) FP16 values (synthetic; no dataset).

Other workloads (--config): long_decode (13 x 8,192), shared_prefix_decode
(64 rows over 125 shared blocks), mixed_prefill (a 4,000-token prompt in
512-token chunks next to 31 decode rows; one step = the whole 8-chunk
schedule, i.e. 8 iterations), gqa_decode (32 rows x 2,300 tokens, 8 K/V heads
serving 32 query heads: 9.65 GB of K/V per step), shared_prefix_cascade (the
shared-prefix workload through cascade decode: the 125 shared blocks are read
once per layer for all 64 rows; roofline on unique bytes), average_decode_int8 (the
headline workload over an 8-bit pool: INT8 codes plus one FP32 scale per
128-value row, 132 bytes per row instead of 256), swap_blocks (a preempted
batch's 384 scattered 8 MB blocks swapped out to page-locked host memory and
back in one launch each; its roofline is a contiguous cudaMemcpyAsync of the
same bytes measured in the same run), mixed_prefill_int8 and mixed_prefill_gqa (the
chunk schedule over an 8-bit pool, and with 8 K/V heads serving 32 query heads).

Rank 0 prints one JSON line. Under torchrun (N > 1) every rank runs its own
replica (weak scaling, no collective on the data path); `value` adds all
ranks' work over the slowest rank's time.

`--impl reference` times the oracle (plain CPU code, oracle/) on the host
cores on a bounded sample of the same workload: one layer per step.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

HEAD_DIM = 128
SCALE = float(np.float32(1.0 / np.sqrt(np.float32(128.0))))


def _iterations(config: str, seed: int = 0):
    """The workload's engine iterations (one for decode configs, 8 for the chunk schedule)."""
    if config in ("average_decode", "average_decode_int8"):
        return [workloads.average_decode(seed)]
    if config == "long_decode":
        return [workloads.long_decode(seed)]
    if config in ("shared_prefix_decode", "shared_prefix_cascade", "shared_prefix_cascade_int8"):
        return [workloads.shared_prefix_decode(seed)]
    if config == "shared_prefix_cascade_gqa":
        w = workloads.shared_prefix_decode(seed, num_blocks=workloads.GQA_POOL_BLOCKS)
        w.num_heads, w.num_q_heads = workloads.GQA_KV_HEADS, workloads.NUM_HEADS
        return [w]
    if config == "gqa_decode":
        return [workloads.gqa_decode(seed)]
    if config in ("mixed_prefill", "mixed_prefill_int8", "mixed_prefill_gqa"):
        first = workloads.mixed_prefill(0, seed=seed)
        its = [workloads.mixed_prefill(c, seed=seed) for c in range(first.meta["num_chunks"])]
        if config == "mixed_prefill_gqa":
            for w in its:
                w.num_heads, w.num_q_heads = workloads.GQA_KV_HEADS, workloads.NUM_HEADS
        return its
    raise KeyError(config)


CONFIG_TEXT = {
    "average_decode": "batch-32 decode, 32 layers x 32 heads x 128 fp16, context = clipped lognormal prompt "
                      "(mean 1,250) + U{0..299} generated + 1, 7,152-block (60 GB) shuffled pool, kv_append of 1 "
                      "token per row",
    "long_decode": "13 rows x 8,192 context tokens, 32 layers, 7,152-block pool, split-K partitions",
    "shared_prefix_decode": "64 rows sharing 125 ref-counted prefix blocks + 1..300 private tokens, 32 layers",
    "mixed_prefill": "one 4,000-token prompt prefilled in 512-token chunks (8 iterations) next to 31 decode rows "
                     "of context U{100..2000} advancing one token per iteration, 32 layers",
    "mixed_prefill_gqa": "the mixed_prefill schedule with 8 K/V heads serving 32 query heads (grouped-query "
                         "attention): a prefill CTA takes 32 tokens of a K/V head's 4 query heads as its 128 rows",
    "mixed_prefill_int8": "the mixed_prefill schedule over an 8-bit pool (INT8 codes, one FP32 scale per (token, "
                          "head) row of K or V): decode rows and prefill chunks both read codes and scales",
    "average_decode_int8": "the average_decode workload over an 8-bit pool (INT8 codes, one FP32 scale per "
                           "(token, head) row of K or V; 2,112-byte tiles), 7,152 blocks (30.9 GB)",
    "shared_prefix_cascade_gqa": "the shared_prefix_cascade workload with 8 K/V heads serving 32 query heads "
                                 "(28,608-block 60 GB pool): a shared-prefix CTA holds 4 rows x 4 query heads",
    "shared_prefix_cascade_int8": "the shared_prefix_cascade workload over an 8-bit pool (INT8 codes, one FP32 "
                                  "scale per (token, head) row of K or V)",
    "shared_prefix_cascade": "64 rows sharing 125 ref-counted prefix blocks + 1..300 private tokens, 32 layers; "
                             "per layer kv_append of the new tokens then cascade decode (shared partitions once "
                             "per group on the tensor cores, the rest per row)",
    "swap_blocks": "swap-out then swap-in of 384 scattered blocks (8,388,608 B each, 3.2 GB) of a 1,024-block "
                   "pool to one page-locked host buffer, one launch each way",
    "gqa_decode": "batch-32 decode at 2,300 context tokens per row, 32 layers, 8 K/V heads serving 32 query heads "
                  "(grouped-query attention, 131,072 B of K/V per token), 28,608-block (60 GB) shuffled pool, "
                  "kv_append of 1 token per row; pool partition 4,096 tokens (one per row)",
}

# The pool's split-K partition length per workload (0: the library's default, 1,024 tokens), the best measured
# on this GB300: the batch-32 MHA rows stream in fewer, longer CTAs at 2,048 (0.951 of HBM peak against 0.926
# at 1,024); the grouped-head workload's 2,300-token rows take one partition each at 4,096, so its 256 CTAs
# run in one wave (0.936 against 0.788 at 1,024: 768 CTAs over 456 resident slots). In the mixed steps the decode
# rows run beside the prefill launch, where shorter CTAs fill the SMs it leaves: the FP16 8-chunk step takes
# 28.50 ms at 768 against 29.13 at 1,024, 29.55 at 512 and 29.59 at 2,048; the 8-bit and grouped-head mixed
# steps are fastest at 1,024 (24.40 and 12.86 ms; 24.56 and 13.03 at 768).
# The plain decode over the shared-prefix workload (64 rows of 2,001-2,300 keys) takes 7.34 ms per step at 2,048
# against 7.95 at 1,024 and 8.05 at 768; its cascade form is fastest at 1,024 (1.99 ms; 2.10 at 768).
CONFIG_PARTITION = {"average_decode": 2048, "long_decode": 2048, "gqa_decode": 4096, "average_decode_int8": 2048,
                    "mixed_prefill": 768, "shared_prefix_decode": 2048, "shared_prefix_cascade_int8": 768,
                    "shared_prefix_cascade_gqa": 768}

CONFIG_DTYPE = {"average_decode_int8": "int8", "mixed_prefill_int8": "int8", "shared_prefix_cascade_int8": "int8"}
SWAP_BLOCKS, SWAP_POOL = 384, 1024

KERNEL_SOURCES = {
    "decode_attn": ["pkv_kernels.cu", "ptx.cuh", "pkv_internal.h"],
    "decode_group_attn": ["pkv_decode_group.cu", "pkv_kernels.cu", "ptx.cuh", "pkv_internal.h"],
    "decode_i8_attn": ["pkv_int8.cu", "ptx.cuh", "pkv_internal.h"],
    "decode_cascade_attn": ["pkv_decode_group.cu", "pkv_kernels.cu", "pkv_int8.cu", "ptx.cuh", "pkv_internal.h"],
    "prefill_attn": ["pkv_prefill.cu", "ptx.cuh", "pkv_internal.h"],
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def _code_only(text: str) -> str:
    """Source text without comments, blank lines and trailing spaces: an edit to comments alone leaves the
    kernel, and so its recorded DRAM traffic, unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def _kernel_source_hash(kernel: str):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_scatter_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def _traffic(kernel: str, config: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's sources are unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(f"{kernel}/{config}")
    if not e or e.get("source_hash") != _kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return parse_clock_lines(self.lines)


def parse_clock_lines(lines):
    sm, smax, power, reasons = [], [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        parts = [x.strip() for x in ln.split(",")]
        if len(parts) < 8:
            continue
        try:
            sm.append(float(parts[0]))
            smax.append(float(parts[1]))
        except ValueError:
            continue
        try:
            power.append(float(parts[2]))
        except ValueError:
            pass
        for name, val in zip(names, parts[4:8]):
            if val.lower().startswith("active"):
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(power) if power else None}


def _gpu_id(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(per_rank_ms, per_rank_units):
    """Whole-job throughput: all ranks' units over the slowest rank's time (seconds)."""
    t = max(per_rank_ms) * 1e-3
    return sum(per_rank_units) / t


def max_over_ranks(values, dist=None, device=None):
    """Element-wise maximum of per-rank timings over the process group; every rank gets the result."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def prefill_pairs(wl) -> int:
    """Unmasked (query, key) pairs of the prefill rows: query at position p sees p + 1 keys."""
    n = 0
    for c, q in zip(wl.ctx_lens[wl.num_decode:], wl.q_lens[wl.num_decode:]):
        lo, hi = int(c) - int(q), int(c)
        n += (lo + 1 + hi) * (hi - lo) // 2
    return n


def row_bytes(dtype: str) -> int:
    """Bytes of one (token, head) row of K or V: 128 FP16 values, or 128 INT8 codes and a 4-byte scale."""
    return HEAD_DIM * 2 if dtype == "fp16" else HEAD_DIM + 4


def kv_bytes(wl, layers, dtype="fp16") -> int:
    """K and V bytes the decode rows read: 2 x heads x row bytes per context token per layer."""
    dec = wl.ctx_lens[:wl.num_decode].astype(np.int64).sum()
    return int(dec) * 2 * wl.num_heads * row_bytes(dtype) * layers


# ------------------------------------------------------------------ ours

def prefill_chunk_summary(chunks, hbm_peak, tf_peak, peak_kind):
    """Roofline of the prefill kernel over a chunk schedule. chunks: (iteration workload, microseconds per
    launch, query heads, K/V heads, bytes per K/V row) per chunk. Each chunk is held against the tensor peak
    (FLOPs of its unmasked (q, k) pairs) and the HBM peak (its K/V prefix read once, q read, out written);
    a chunk whose FLOPs per byte sit below the ridge tf_peak / hbm_peak is HBM-bound."""
    per, fl_tot, us_tot = [], 0.0, 0.0
    fl_t, us_t = 0.0, 0.0  # the tensor-bound chunks only
    ridge = tf_peak * 1e12 / (hbm_peak * 1e9)
    for wl, us, hq, hkv, rb in chunks:
        fl = 4 * HEAD_DIM * hq * prefill_pairs(wl)
        B = wl.num_decode
        by = sum(int(c) * 2 * hkv * rb + 2 * int(q) * hq * HEAD_DIM * 2
                 for c, q in zip(wl.ctx_lens[B:], wl.q_lens[B:]))
        tf = fl / (us * 1e-6) / 1e12
        gbs = by / (us * 1e-6) / 1e9
        per.append({"chunk": int(wl.meta.get("chunk", len(per))), "us": round(us, 2), "tflops": round(tf, 1),
                    "frac": round(tf / tf_peak, 4), "gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
                    "bound": "tensor" if fl / by >= ridge else "hbm"})
        fl_tot += fl
        us_tot += us
        if fl / by >= ridge:
            fl_t += fl
            us_t += us
    agg = fl_tot / (us_tot * 1e-6) / 1e12
    agg_t = fl_t / (us_t * 1e-6) / 1e12 if us_t > 0 else None
    return {"bound": "tensor", "achieved": round(agg, 1), "peak": tf_peak,
            "peak_kind": peak_kind + " bf16 dense (fp16 runs at the same rate)", "unit": "TFLOP/s",
            "frac": round(agg / tf_peak, 4),
            "aggregate": {"chunks": len(per), "us_per_layer": round(us_tot, 2), "tflops": round(agg, 1),
                          "frac": round(agg / tf_peak, 4)},
            "aggregate_tensor_bound": {"chunks": sum(1 for c in per if c["bound"] == "tensor"),
                                       "us_per_layer": round(us_t, 2),
                                       "tflops": round(agg_t, 1) if agg_t is not None else None,
                                       "frac": round(agg_t / tf_peak, 4) if agg_t is not None else None},
            "per_chunk": per}


def prefill_schedule(torch, pkv, pool, L, dev, gen, steps, stream, hbm_peak, tf_peak, peak_kind):
    """The prefill kernel alone over the 4,000-token prompt's 8-chunk schedule (the mixed_prefill workload's
    prefill rows, 32 heads), on this run's pool: per chunk a CUDA graph of its L per-layer launches, replayed
    `steps` times between two events on the launching stream; per-launch time = elapsed / (steps x L)."""
    iters = _iterations("mixed_prefill")
    datas = [StepData(torch, pkv, pool, wl, m, L, dev, gen) for wl, m in zip(iters, _metadata(pkv, iters))]
    graphs = []
    for d in datas:
        tables_d, ctx_d, qs_d, _ = d.dev
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
            for l in range(L):
                pool.prefill_attn(l, d.q[l], qs_d[d.B:], tables_d[d.B:], ctx_d[d.B:], d.max_q, SCALE, d.out[l],
                                  torch.cuda.current_stream(dev))
        graphs.append(g)
    torch.cuda.synchronize(dev)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in graphs]
    for (a, b), g in zip(ev, graphs):
        a.record(stream)
        for _ in range(steps):
            g.replay()
        b.record(stream)
    torch.cuda.synchronize(dev)
    st, flags = pool.get_status(stream)
    if st != pkv.PKV_OK:
        raise RuntimeError(f"device status {st} flags {flags:#x}")
    chunks = [(d.wl, a.elapsed_time(b) * 1e3 / (steps * L), d.wl.q_heads, d.wl.num_heads, row_bytes("fp16"))
              for d, (a, b) in zip(datas, ev)]
    res = prefill_chunk_summary(chunks, hbm_peak, tf_peak, peak_kind)
    res["kernel"] = "prefill_kernel (tcgen05)"
    res["workload"] = ("the mixed_prefill schedule's prefill rows: a 4,000-token prompt in 512-token chunks, "
                       "32 layers x 32 heads x 128, on this run's 7,152-block pool")
    res["timing"] = ("CUDA events around a graph of one chunk's prefill launches for all layers, replayed; "
                     "per-launch = elapsed / (replays x layers)")
    return res



class StepData:
    """Device metadata and per-layer tensors of one engine iteration."""

    def __init__(self, torch, pkv, pool, wl, meta, layers, dev, gen):
        tables, ctx, slots, qs = meta
        self.wl = wl
        self.host = [torch.from_numpy(np.ascontiguousarray(x)).pin_memory() for x in (tables, ctx, qs, slots)]
        self.dev = [x.to(dev) for x in self.host]
        T, H, Hq = wl.num_tokens, wl.num_heads, wl.q_heads
        self.q = torch.randn((layers, T, Hq, HEAD_DIM), generator=gen, device=dev).half()
        self.k = torch.randn((layers, T, H, HEAD_DIM), generator=gen, device=dev).half()
        self.v = torch.randn((layers, T, H, HEAD_DIM), generator=gen, device=dev).half()
        self.out = torch.empty_like(self.q)
        B = wl.num_decode
        self.B = B
        self.max_q = int(wl.q_lens[B:].max()) if wl.num_seqs > B else 0
        stride, qstride = T * H * HEAD_DIM, T * Hq * HEAD_DIM
        tables_d, ctx_d, qs_d, slots_d = self.dev
        self.desc = pkv.make_step_desc(num_decode=B, num_prefill=wl.num_seqs - B, num_tokens=T, max_q_len=self.max_q,
                                       max_blocks=tables.shape[1], first_layer=0, num_layers=layers, scale=SCALE,
                                       block_tables=tables_d, ctx_lens=ctx_d, q_start_loc=qs_d, slot_mapping=slots_d,
                                       q=self.q, k=self.k, v=self.v, out=self.out, q_layer_stride=qstride,
                                       k_layer_stride=stride, v_layer_stride=stride, out_layer_stride=qstride)
        self.ws_bytes = pool.step_workspace_bytes(self.desc)
        # the iteration's decode rows alone, over all layers, as pkv_step runs them (one counter clear, then the
        # layers' decode launches chained with programmatic dependencies): the per-kernel timing of decode
        self.dec_desc = self.desc if wl.num_seqs == B else (
            pkv.make_step_desc(num_decode=B, num_prefill=0, num_tokens=B, max_q_len=0, max_blocks=tables.shape[1],
                               first_layer=0, num_layers=layers, scale=SCALE, block_tables=tables_d,
                               ctx_lens=ctx_d, q_start_loc=qs_d, slot_mapping=slots_d, q=self.q, k=self.k, v=self.v,
                               out=self.out, q_layer_stride=qstride, k_layer_stride=stride, v_layer_stride=stride,
                               out_layer_stride=qstride) if B else None)
        # one-layer steps (same kernels as the full step) for per-launch timing of decode-only iterations without
        # graphs
        self.layer_desc = [
            pkv.make_step_desc(num_decode=B, num_prefill=0, num_tokens=T, max_q_len=0, max_blocks=tables.shape[1],
                               first_layer=l, num_layers=1, scale=SCALE, block_tables=tables_d, ctx_lens=ctx_d,
                               q_start_loc=qs_d, slot_mapping=slots_d, q=self.q[l], k=self.k[l], v=self.v[l],
                               out=self.out[l], q_layer_stride=qstride, k_layer_stride=stride,
                               v_layer_stride=stride, out_layer_stride=qstride)
            for l in range(layers)] if wl.num_seqs == B else None


def _metadata(pkv, iterations):
    """Step metadata from libpkv's block manager, iteration after iteration, as a serving loop gets it.

    Blocks are handed out in the order of the first iteration's tables (a
    random permutation of the pool), so for a single decode iteration the
    tables equal the workload's own."""
    wl0 = iterations[0]
    seen = []
    for r in range(wl0.num_seqs):
        seen.extend(int(b) for b in wl0.block_tables[r] if b >= 0)
    order = list(dict.fromkeys(seen))
    rest = np.setdiff1d(np.arange(wl0.num_blocks), np.array(order, np.int64))
    mgr = pkv.Pool(None, wl0.num_blocks, num_layers=wl0.num_layers, num_heads=wl0.num_heads,
                   free_order=np.concatenate([np.array(order, np.int64), rest]))
    prefix = int(wl0.meta.get("prefix_blocks", 0))
    if prefix:
        assert mgr.seq_grow(-1, prefix * 16) == pkv.PKV_OK
        for r in range(wl0.num_seqs):
            assert mgr.seq_share_prefix(r, -1, prefix) == pkv.PKV_OK
    out = []
    for wl in iterations:
        for r in range(wl.num_seqs):
            assert mgr.seq_grow(r, int(wl.ctx_lens[r])) == pkv.PKV_OK
        st, tables, ctx, slots, qs = mgr.build_step(np.arange(wl.num_seqs), wl.q_lens, wl0.max_blocks)
        assert st == pkv.PKV_OK and np.array_equal(ctx, wl.ctx_lens)
        out.append((tables, ctx, slots, qs))
    if len(iterations) == 1 and not prefix:
        assert np.array_equal(out[0][0], wl0.block_tables)
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist
    import paged_kv_cache_scatter_gb300 as pkv
    from paged_kv_cache_scatter_gb300 import build as pkv_build

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pkv_build.build()
    pkv.load()

    iters = _iterations(args.config, args.seed)
    wl0 = iters[0]
    L = args.layers or wl0.num_layers
    H, Hq = wl0.num_heads, wl0.q_heads
    dtype = CONFIG_DTYPE.get(args.config, "fp16")
    dev = torch.device("cuda", local)

    if dtype == "int8":
        pool_t = torch.empty(pkv.Pool.bytes_needed(wl0.num_blocks, L, H, "int8"), dtype=torch.uint8, device=dev)
        workloads.fill_int8_tiles_(pool_t, workloads.value_seed(wl0.seed, "pool"))
    else:
        pool_t = torch.empty(workloads.pool_shape(wl0.num_blocks, L, H), dtype=torch.float16, device=dev)
        workloads.fill_normal_fp16_(pool_t, workloads.value_seed(wl0.seed, "pool"))
    if not args.partition_tokens:
        args.partition_tokens = CONFIG_PARTITION.get(args.config, 0)
    pool = pkv.Pool(pool_t, wl0.num_blocks, num_layers=L, num_heads=H, partition_tokens=args.partition_tokens,
                    num_q_heads=Hq, dtype=dtype)
    gen = torch.Generator(device=dev)
    gen.manual_seed(workloads.value_seed(wl0.seed, "q"))
    steps = [StepData(torch, pkv, pool, wl, m, L, dev, gen) for wl, m in zip(iters, _metadata(pkv, iters))]
    wspace = torch.empty(max(max(s.ws_bytes for s in steps), 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    cascade = args.config.startswith("shared_prefix_cascade")
    if cascade:
        s0 = steps[0]
        need = pool.decode_cascade_workspace_bytes(s0.B, s0.desc.max_blocks)
        if need > wspace.numel():
            wspace = torch.empty(need, dtype=torch.uint8, device=dev)
        gs, gb, widest = pkv.cascade_groups(s0.host[0].numpy(), s0.host[1].numpy())
        groups = (torch.from_numpy(gs).to(dev), torch.from_numpy(gb).to(dev), widest)

    def step(strm=None):
        strm = strm if strm is not None else stream
        for s in steps:
            if cascade:
                tables_d, ctx_d, _, slots_d = s.dev
                for l in range(L):
                    pool.kv_append(l, s.k[l], s.v[l], slots_d, strm)
                    pool.decode_attn_cascade(l, s.q[l], tables_d, ctx_d, groups, SCALE, s.out[l], wspace, strm)
            else:
                pool.step(s.desc, wspace, strm)

    def check_status():
        st, flags = pool.get_status(stream)
        if st != pkv.PKV_OK:
            raise RuntimeError(f"device status {st} flags {flags:#x}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    check_status()

    # The timed step is a CUDA graph of the whole iteration (all layers), as a serving loop would replay it.
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap, capture_error_mode="thread_local"):
            step(torch.cuda.current_stream(dev))
        torch.cuda.synchronize(dev)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize(dev)
        check_status()

    has_prefill = any(s.max_q for s in steps)
    has_decode = any(s.B for s in steps)
    kv_step = sum(kv_bytes(s.wl, L, dtype) for s in steps)
    pairs_step = sum(prefill_pairs(s.wl) for s in steps) * L
    flops_step = 4 * HEAD_DIM * Hq * pairs_step
    tokens_step = sum(int(s.wl.ctx_lens[:s.B].astype(np.int64).sum()) for s in steps) * L
    launches_step = 0
    for s in steps:
        # per layer: decode (it also appends the decode rows' K/V); kv_append + prefill for chunk rows
        per_layer = (1 if s.B else 0) + (2 if s.max_q else 0) + (2 if cascade else 0)
        launches_step += per_layer * L

    sampler = ClockSampler(_gpu_id(torch, local))
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    # ---- timed region 1: the whole step through pkv_step
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = ev(), ev()
    marks = [ev() for _ in range(args.steps)]  # one event after each step: the per-step distribution
    e0.record(stream)
    for i in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step()
        marks[i].record(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    t_ms = e0.elapsed_time(e1)
    step_times = [(e0 if i == 0 else marks[i - 1]).elapsed_time(marks[i]) for i in range(args.steps)]

    # ---- timed region 2: each attention kernel alone. With graphs (the default), one CUDA graph per iteration
    # and kernel holds that kernel's launches for all layers, replayed between two events: per-launch time =
    # elapsed / layers, the kernel back to back with itself as the step graph runs it. (Events around single
    # stream launches would also time the stream's launch gaps, several microseconds per launch on this
    # platform.) With --no-graph: events around every call.
    def launch_dec(s, l, strm):
        tables_d, ctx_d, qs_d, slots_d = s.dev
        if cascade:
            pool.decode_attn_cascade(l, s.q[l], tables_d, ctx_d, groups, SCALE, s.out[l], wspace, strm)
        elif s.layer_desc is not None:
            # decode-only: the one-layer step is exactly the fused decode+append launch of the full step
            pool.step(s.layer_desc[l], wspace, strm)
        else:
            pool.decode_attn(l, s.q[l, :s.B], tables_d[:s.B], ctx_d[:s.B], SCALE, s.out[l, :s.B], wspace, strm)

    def launch_pre(s, l, strm):
        tables_d, ctx_d, qs_d, slots_d = s.dev
        pool.prefill_attn(l, s.q[l], qs_d[s.B:], tables_d[s.B:], ctx_d[s.B:], s.max_q, SCALE, s.out[l], strm)

    dec_ev, pre_ev = [], []  # (start event, end event, iteration, launches between them)
    torch.cuda.synchronize(dev)
    if graph is not None:
        kgraphs = []
        for s in steps:
            pair = []
            for use, fn in ((bool(s.B) or cascade, launch_dec), (bool(s.max_q), launch_pre)):
                g = None
                if use:
                    g = torch.cuda.CUDAGraph()
                    cap = torch.cuda.Stream(dev)
                    cap.wait_stream(stream)
                    with torch.cuda.graph(g, stream=cap, capture_error_mode="thread_local"):
                        if fn is launch_dec and not cascade:
                            # all layers' decode launches as pkv_step issues them: one counter clear, then the
                            # layers chained with programmatic dependencies
                            pool.step(s.dec_desc, wspace, torch.cuda.current_stream(dev))
                        else:
                            for l in range(L):
                                fn(s, l, torch.cuda.current_stream(dev))
                pair.append(g)
            kgraphs.append(pair)
        torch.cuda.synchronize(dev)
        for s, (gd, gp) in zip(steps, kgraphs):  # one untimed replay each
            for g in (gd, gp):
                if g is not None:
                    g.replay()
        torch.cuda.synchronize(dev)
        for _ in range(args.steps):
            for s, (gd, gp) in zip(steps, kgraphs):
                for g, lst in ((gd, dec_ev), (gp, pre_ev)):
                    if g is None:
                        continue
                    a, b = ev(), ev()
                    a.record(stream)
                    g.replay()
                    b.record(stream)
                    lst.append((a, b, s, L))
    else:
        for _ in range(args.steps):
            for s in steps:
                for l in range(L):
                    if cascade or s.layer_desc is None:  # a decode-only layer step appends inside its launch
                        pool.kv_append(l, s.k[l], s.v[l], s.dev[3], stream)
                    for use, fn, lst in ((bool(s.B) or cascade, launch_dec, dec_ev), (bool(s.max_q), launch_pre, pre_ev)):
                        if use:
                            a, b = ev(), ev()
                            a.record(stream)
                            fn(s, l, stream)
                            b.record(stream)
                            lst.append((a, b, s, 1))
    torch.cuda.synchronize(dev)
    hbm_peak, tf_peak, peak_kind = _peaks()
    sched_roofline = None
    if args.config == "average_decode" and not args.no_prefill_schedule and L == wl0.num_layers:
        # the prefill kernel over the mixed workload's 8-chunk schedule, on this run's pool, inside the clock
        # record (an extra key of the line: the headline stays decode)
        sched_roofline = prefill_schedule(torch, pkv, pool, L, dev, gen, args.steps, stream, hbm_peak, tf_peak,
                                          peak_kind)
    clocks = sampler.stop()
    check_status()
    dec_ms = sum(a.elapsed_time(b) for a, b, _, _ in dec_ev)
    pre_ms = sum(a.elapsed_time(b) for a, b, _, _ in pre_ev)

    # ---- end to end: host buffers in, host result out, every step. As a serving loop runs it: two sets of
    # device buffers, the next step's host-to-device copies (one stream) and this step's result read back (a
    # second stream) run beside the step's kernels, ordered by events (a set's inputs are overwritten only once
    # the step that used them and its read-back are done).
    host_io = []
    for s in steps:
        host_io.append([(x.cpu().pin_memory(), x) for x in (s.q, s.k, s.v)] + list(zip(s.host, s.dev)))
    outs_h = [torch.empty(s.out.shape, dtype=s.out.dtype).pin_memory() for s in steps]
    twins = [StepData(torch, pkv, pool, s.wl, m, L, dev, gen) for s, m in zip(steps, _metadata(pkv, iters))]
    sets = [[(s, [(src, dst) for (src, _), dst in zip(io, [s.q, s.k, s.v] + list(s.dev))], oh)
             for s, io, oh in zip(st, host_io, outs_h)] for st in (steps, twins)]

    def run_unit(t):  # one iteration of the step on one buffer set
        if cascade:
            tables_d, ctx_d, _, slots_d = t.dev
            for l in range(L):
                pool.kv_append(l, t.k[l], t.v[l], slots_d, stream)
                pool.decode_attn_cascade(l, t.q[l], tables_d, ctx_d, groups, SCALE, t.out[l], wspace, stream)
        else:
            pool.step(t.desc, wspace, stream)

    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n_units = 2 * len(steps)
    in_ready = [ev() for _ in range(n_units)]
    done = [ev() for _ in range(n_units)]
    read = [ev() for _ in range(n_units)]
    e4, e5 = ev(), ev()
    torch.cuda.synchronize(dev)
    e4.record(stream)
    h2d_s.wait_stream(stream)
    d2h_s.wait_stream(stream)
    k = 0
    for _ in range(args.steps):
        for si in range(len(steps)):
            u = (k % 2) * len(steps) + si  # buffer set k % 2 of iteration si
            t, tio, toh = sets[k % 2][si]
            h2d_s.wait_event(done[u])  # the set's previous step is done with its inputs
            with torch.cuda.stream(h2d_s):
                for src, dst in tio:
                    dst.copy_(src, non_blocking=True)
            in_ready[u].record(h2d_s)
            stream.wait_event(in_ready[u])
            stream.wait_event(read[u])  # its previous result has been read back
            run_unit(t)
            done[u].record(stream)
            d2h_s.wait_event(done[u])
            with torch.cuda.stream(d2h_s):
                toh.copy_(t.out, non_blocking=True)
            read[u].record(d2h_s)
        k += 1
    stream.wait_stream(h2d_s)
    stream.wait_stream(d2h_s)
    e5.record(stream)
    torch.cuda.synchronize(dev)
    check_status()
    e2e_ms = e4.elapsed_time(e5)
    h2d = sum(src.numel() * src.element_size() for io in host_io for src, _ in io)
    d2h = sum(o.numel() * o.element_size() for o in outs_h)

    t_ms, e2e_ms = max_over_ranks([t_ms, e2e_ms], dist if ws > 1 else None, dev)

    K = args.steps
    if has_decode:
        metric = "decode KV GB/s (KV bytes read per 32-layer iteration / iteration time) at batch 32"
        value = kv_step * K * ws / (t_ms * 1e-3) / 1e9
        unit = "GB/s"
        e2e_value = kv_step * K * ws / (e2e_ms * 1e-3) / 1e9
    else:
        metric = "prefill attention TFLOP/s"
        value = flops_step * K * ws / (t_ms * 1e-3) / 1e12
        unit = "TFLOP/s"
        e2e_value = flops_step * K * ws / (e2e_ms * 1e-3) / 1e12
    n_dec = sum(n for *_, n in dec_ev)
    n_pre = sum(n for *_, n in pre_ev)
    # K/V context read + q read + out written, per launch
    dec_bytes_launch = (kv_step / L / len(steps)) + sum(2 * s.B * Hq * HEAD_DIM * 2 for s in steps) / len(steps)
    dec_kernel = "decode_kernel" if Hq == H else "decode_group_kernel (mma.sync m16n8k16, one K/V read per group)"
    dec_src = "decode_attn" if Hq == H else "decode_group_attn"
    if dtype == "int8":
        dec_kernel, dec_src = "decode_i8_kernel (INT8 codes dequantised in the loaders)", "decode_i8_attn"
    unique_step = None
    if args.config.startswith("shared_prefix"):
        # K/V bytes a layer must read at least once: the shared prefix once, then each row's own tokens
        w0 = steps[0].wl
        pre = int(w0.meta["prefix_blocks"]) * 16
        unique_tok = pre + int((w0.ctx_lens[:w0.num_decode].astype(np.int64) - pre).sum())
        unique_step = unique_tok * 2 * H * row_bytes(dtype) * L
    if cascade:
        if dtype == "int8":
            dec_kernel = ("cascade decode over an 8-bit pool: decode_i8_kernel<true, true> (shared partitions, 16 "
                          "query rows per CTA, mma.sync) then decode_i8_kernel (the rest, merge)")
        elif Hq != H:
            dec_kernel = ("cascade decode, grouped heads: decode_group_kernel<true, true> (shared partitions, 4 rows x "
                          "4 query heads per CTA, mma.sync) then decode_group_kernel (the rest, merge)")
        else:
            dec_kernel = ("cascade decode: decode_group_kernel<true, true> (shared partitions, 16 rows per CTA, "
                          "mma.sync) then decode_kernel (the rest, merge)")
        dec_src = "decode_cascade_attn"
        # the roofline of a cascade launch: unique bytes + q and out
        dec_bytes_launch = unique_step / L / len(steps) + sum(2 * s.B * Hq * HEAD_DIM * 2 for s in steps) / len(steps)
    rooflines = {}
    if n_dec:
        ach = dec_bytes_launch / (dec_ms / n_dec * 1e-3) / 1e9
        rooflines["decode"] = {"bound": "hbm",
                               "kernel": dec_kernel + " (with its split-K merge; decode-only steps: also the "
                                         "decode rows' kv_append), incl. the workspace counter clear",
                               "achieved": round(ach, 1), "peak": hbm_peak, "peak_kind": peak_kind, "unit": "GB/s",
                               "frac": round(ach / hbm_peak, 4),
                               "traffic": _traffic(dec_src, args.config),
                               "algorithmic_bytes_per_launch": int(dec_bytes_launch),
                               "avg_launch_us": round(dec_ms / n_dec * 1e3, 2)}
    if pre_ev:
        fl = 4 * HEAD_DIM * Hq * sum(prefill_pairs(s.wl) * n for _, _, s, n in pre_ev)
        pre_kernel = ("prefill_kernel<8-bit> (tcgen05; codes by TMA become FP16 in shared memory, row scales "
                      "applied in the softmax)" if dtype == "int8" else "prefill_kernel (tcgen05)")
        chunks = []
        for s in steps:
            if s.max_q:
                us = (sum(a.elapsed_time(b) for a, b, s2, _ in pre_ev if s2 is s)
                      / max(1, sum(n for _, _, s2, n in pre_ev if s2 is s)) * 1e3)
                chunks.append((s.wl, us, Hq, H, row_bytes(dtype)))
        rooflines["prefill"] = prefill_chunk_summary(chunks, hbm_peak, tf_peak, peak_kind)
        rooflines["prefill"].update({"kernel": pre_kernel, "traffic": _traffic("prefill_attn", args.config),
                                     "algorithmic_flops_per_launch": int(fl / n_pre),
                                     "avg_launch_us": round(pre_ms / n_pre * 1e3, 2)})
    kernel_timing = ("CUDA events around a graph of one kernel's launches for all layers, per-launch = elapsed / "
                     "layers" if graph is not None else "CUDA events around every launch")
    for r in rooflines.values():
        r["timing"] = kernel_timing
    if sched_roofline is not None:
        rooflines["prefill"] = sched_roofline
    dominant = "decode" if (dec_ms >= pre_ms and n_dec) else "prefill"

    result = {
        "metric": metric,
        "value": round(value, 1),
        "unit": unit,
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(t_ms / K, 4),
        "step_ms": {"p10": round(float(np.percentile(step_times, 10)), 4),
                    "median": round(float(np.median(step_times)), 4),
                    "p90": round(float(np.percentile(step_times, 90)), 4)},
        "us_per_iteration": round(t_ms / K / len(steps) * 1e3, 1),
        "attention_tokens_per_s": round(tokens_step * K * ws / (t_ms * 1e-3), 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 storage, f32 arithmetic" if dtype == "fp16" else "int8 storage (fp32 scales), f32 arithmetic",
        "data": "synthetic",
        "config": {"workload": args.config, "description": CONFIG_TEXT[args.config], "num_layers": L,
                   "iterations_per_step": len(steps), "num_seqs": wl0.num_seqs, "heads": H, "query_heads": Hq,
                   "kv_dtype": dtype,
                   "head_dim": HEAD_DIM,
                   "pool_blocks": wl0.num_blocks, "kv_bytes_per_step": kv_step,
                   "prefill_flops_per_step": flops_step, "seed": wl0.seed,
                   "partition_tokens": args.partition_tokens or 1024,
                   "max_context": int(max(int(s.wl.ctx_lens.max()) for s in steps)),
                   "l2": "inputs larger than L2 (every step reads the whole KV context of all layers)",
                   "cuda_graph": graph is not None},
        "clocks": clocks,
        "gpu_launches": launches_step * K,
        "roofline": rooflines[dominant],
        "rooflines": rooflines,
        "e2e": {"value": round(e2e_value, 1), "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms / K, 4),
                "how": ("the step with every step's inputs copied from pinned host memory and its result read back "
                        "inside the timed region; the next step's copies and this step's read-back on two streams "
                        "of their own beside the step's kernels (two sets of device buffers)")},
    }
    if has_decode:
        result["hbm_frac_of_measured_peak"] = round(value / hbm_peak, 4)
    if unique_step:
        result["unique_kv_bytes_per_step"] = unique_step
        result["unique_gbs"] = round(unique_step * K * ws / (t_ms * 1e-3) / 1e9, 1)
        result["unique_frac_of_measured_peak"] = round(unique_step * K * ws / (t_ms * 1e-3) / 1e9 / hbm_peak, 4)
    if has_prefill:
        result["prefill_tflops"] = round(flops_step * K * ws / (t_ms * 1e-3) / 1e12, 1)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(iters[0], pool_t, args.cpu_seconds, L, dtype)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------ swap

def run_swap(args):
    """Block swap out + in through pkv_swap_blocks_out / _in; the link's own rate from cudaMemcpyAsync."""
    import torch
    import torch.distributed as dist
    import paged_kv_cache_scatter_gb300 as pkv
    from paged_kv_cache_scatter_gb300 import build as pkv_build

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    pkv_build.build()
    pkv.load()
    dev = torch.device("cuda", local)
    L, H, N, n = 32, 32, SWAP_POOL, SWAP_BLOCKS
    pool_t = torch.empty(workloads.pool_shape(N, L, H), dtype=torch.float16, device=dev)
    workloads.fill_normal_fp16_(pool_t, workloads.value_seed(args.seed, "pool"))
    pool = pkv.Pool(pool_t, N, num_layers=L, num_heads=H)
    bb = pkv.Pool.bytes_needed(1, L, H)
    rng = np.random.default_rng(args.seed)
    blocks = torch.from_numpy(rng.choice(N, n, replace=False).astype(np.int32)).to(dev)
    pairs = torch.from_numpy(np.stack([rng.choice(N // 2, n // 4, replace=False),
                                       N // 2 + rng.choice(N // 2, n // 4, replace=False)], 1).astype(np.int32)).to(dev)
    host = torch.empty(n * bb, dtype=torch.uint8).pin_memory()
    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step():
        pool.swap_blocks_out(blocks, host, stream)
        pool.swap_blocks_in(blocks, host, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st, flags = pool.get_status(stream)
    if st != pkv.PKV_OK:
        raise RuntimeError(f"device status {st} flags {flags:#x}")
    sampler = ClockSampler(_gpu_id(torch, local))
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    e0, e1, e2, e3 = ev(), ev(), ev(), ev()
    e0.record(stream)
    for _ in range(args.steps):
        pool.swap_blocks_out(blocks, host, stream)
    e1.record(stream)
    for _ in range(args.steps):
        pool.swap_blocks_in(blocks, host, stream)
    e2.record(stream)
    torch.cuda.synchronize(dev)
    t_out, t_in = e0.elapsed_time(e1), e1.elapsed_time(e2)
    # the link's rate for the same bytes, contiguous, through the copy engines
    flat = pool_t.view(-1)[: n * bb // 2].view(torch.uint8)
    c0, c1, c2 = ev(), ev(), ev()
    c0.record(stream)
    for _ in range(args.steps):
        host.copy_(flat, non_blocking=True)
    c1.record(stream)
    for _ in range(args.steps):
        flat.copy_(host, non_blocking=True)
    c2.record(stream)
    # copy-on-write block copies inside HBM
    k0, k1 = ev(), ev()
    k0.record(stream)
    for _ in range(args.steps):
        pool.copy_blocks(pairs, stream)
    k1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    st, flags = pool.get_status(stream)
    if st != pkv.PKV_OK:
        raise RuntimeError(f"device status {st} flags {flags:#x}")
    m_out, m_in, t_cow = c0.elapsed_time(c1), c1.elapsed_time(c2), k0.elapsed_time(k1)
    t_ms = max_over_ranks([t_out + t_in], dist if ws > 1 else None, dev)[0]
    K = args.steps
    moved = 2 * n * bb * K
    value = moved * ws / (t_ms * 1e-3) / 1e9
    link = moved / ((m_out + m_in) * 1e-3) / 1e9
    hbm_peak, _, peak_kind = _peaks()
    cow_gbs = 2 * pairs.shape[0] * bb * K / (t_cow * 1e-3) / 1e9
    # end to end through the public calls: the block list comes from host memory each step, and the
    # host copy is read back after the round trip (it is the data)
    blocks_h = blocks.cpu().pin_memory()
    x0, x1 = ev(), ev()
    torch.cuda.synchronize(dev)
    x0.record(stream)
    for _ in range(K):
        blocks.copy_(blocks_h, non_blocking=True)
        step()
    x1.record(stream)
    torch.cuda.synchronize(dev)
    e2e = moved / (x0.elapsed_time(x1) * 1e-3) / 1e9
    result = {
        "metric": "block swap GB/s (bytes moved out to page-locked host memory and back in / time)",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(t_ms / K, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bytes (f16 pool)", "data": "synthetic",
        "config": {"workload": "swap_blocks", "description": CONFIG_TEXT["swap_blocks"], "blocks": n,
                   "block_bytes": bb, "pool_blocks": N, "l2": "3.2 GB per direction, above the 129 MB L2"},
        "out_gbs": round(n * bb * K / (t_out * 1e-3) / 1e9, 1), "in_gbs": round(n * bb * K / (t_in * 1e-3) / 1e9, 1),
        "clocks": clocks, "gpu_launches": 2 * K,
        "roofline": {"bound": "c2c", "achieved": round(value, 1), "peak": round(link, 1),
                     "peak_kind": "measured in this run: cudaMemcpyAsync of the same bytes, contiguous, "
                                  "device to pinned host and back", "unit": "GB/s", "frac": round(value / link, 4),
                     "traffic": None},
        "copy_blocks": {"gbs": round(cow_gbs, 1), "pairs": int(pairs.shape[0]),
                        "frac_of_hbm": round(cow_gbs / hbm_peak, 4), "peak_kind": peak_kind,
                        "note": "copy-on-write block copies inside HBM, read + write bytes per second"},
        "e2e": {"value": round(e2e, 1), "unit": "GB/s", "h2d_bytes_per_step": int(n * 4 + n * bb),
                "d2h_bytes_per_step": int(n * bb)},
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        hb = np.empty(0)
        g = oracle.geom(64, L, H)
        mini = np.zeros(oracle.pool_bytes(g) // 2, np.uint16)
        bl = np.arange(48, dtype=np.int32)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < min(args.cpu_seconds, 5.0):
            hb = oracle.swap_out(mini, g, bl)
            oracle.swap_in(mini, g, bl, hb)
            reps += 1
        dt = time.perf_counter() - t0
        result["cpu_baseline"] = {"value": round(2 * len(bl) * bb * reps / dt / 1e9, 2), "unit": "GB/s", "cores": 1,
                                  "kind": "oracle", "sample": f"48 blocks out and in, {reps} round trips, host memory"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------ oracle timings

def _layer_sample(wl, layer, pool_t=None, seed=0, dtype="fp16"):
    """Host mini-pool of one layer's referenced blocks (renumbered), its tables and q."""
    import torch
    nb = -(-wl.ctx_lens.astype(np.int64) // 16)
    ids = np.concatenate([wl.block_tables[r, :nb[r]] for r in range(wl.num_seqs)]).astype(np.int64)
    uniq, inv = np.unique(ids, return_inverse=True)
    if dtype == "int8":
        layer_bytes = 2 * wl.num_heads * 2112
        if pool_t is not None:
            blocks = pool_t.view(wl.num_blocks, -1, layer_bytes)
            sub = blocks.index_select(0, torch.from_numpy(uniq).to(pool_t.device))[:, layer].contiguous()
            mini = sub.cpu().numpy().reshape(-1)
        else:
            t = torch.empty(len(uniq) * layer_bytes, dtype=torch.uint8)
            mini = workloads.fill_int8_tiles_(t, seed + layer).numpy()
    elif pool_t is not None:
        sub = pool_t.index_select(0, torch.from_numpy(uniq).to(pool_t.device))[:, layer:layer + 1].contiguous()
        mini = sub.cpu().view(torch.int16).numpy().view(np.uint16)
    else:
        shape = workloads.pool_shape(len(uniq), 1, wl.num_heads)
        mini = workloads.normal_fp16(shape, seed + layer).numpy().view(np.uint16)
    tables = np.full_like(wl.block_tables, -1)
    cur = 0
    for r in range(wl.num_seqs):
        tables[r, :nb[r]] = inv[cur:cur + nb[r]]
        cur += nb[r]
    q = workloads.normal_fp16((wl.num_tokens, wl.q_heads, HEAD_DIM),
                              workloads.value_seed(wl.seed, "q", layer)).numpy()
    return np.ascontiguousarray(mini), tables, q.view(np.uint16), len(uniq)


def _oracle_layer(oracle, wl, mini, tables, q, n, dtype="fp16"):
    g = oracle.geom(n, 1, wl.num_heads, num_q_heads=wl.q_heads, dtype=oracle.INT8 if dtype == "int8" else oracle.FP16)
    B = wl.num_decode
    if B:
        oracle.decode_attn(mini, g, 0, q[:B], tables[:B], wl.ctx_lens[:B], SCALE)
    if wl.num_seqs > B:
        oracle.prefill_attn(mini, g, 0, q, wl.q_start_loc()[B:], tables[B:], wl.ctx_lens[B:], SCALE)


def cpu_baseline(wl, pool_t, budget_s, layers, dtype="fp16"):
    import oracle
    threads = len(os.sched_getaffinity(0))
    oracle.set_num_threads(threads)
    t_total, done = 0.0, 0
    for layer in range(layers):
        mini, tables, q, n = _layer_sample(wl, layer, pool_t, dtype=dtype)
        t0 = time.perf_counter()
        _oracle_layer(oracle, wl, mini, tables, q, n, dtype)
        t_total += time.perf_counter() - t0
        done += 1
        if t_total >= budget_s:
            break
    kv = kv_bytes(wl, done, dtype)
    res = {"unit": "GB/s", "cores": threads, "kind": "oracle", "seconds": round(t_total, 2),
           "sample": f"all rows and heads of the first iteration for {done} of {layers} layers (referenced blocks "
                     f"copied to host first, copy not timed)"}
    if wl.num_decode:
        res["value"] = round(kv / t_total / 1e9, 3)
    else:
        res["unit"] = "TFLOP/s"
        res["value"] = round(4 * HEAD_DIM * wl.q_heads * prefill_pairs(wl) * done / t_total / 1e12, 6)
    return res


def run_reference(args):
    ws, rank, local = _dist()
    if rank != 0:
        return
    import oracle
    if args.config == "swap_blocks":
        g = oracle.geom(64, 32, 32)
        mini = np.zeros(oracle.pool_bytes(g) // 2, np.uint16)
        bl = np.arange(48, dtype=np.int32)
        bb = oracle.bytes_per_block(g)
        times = []
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            hb = oracle.swap_out(mini, g, bl)
            oracle.swap_in(mini, g, bl, hb)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        value = 2 * len(bl) * bb * len(times) / sum(times) / 1e9
        print(json.dumps({"impl": "reference", "metric": "block swap GB/s (bytes moved out to page-locked host "
                          "memory and back in / time)", "value": round(value, 3), "unit": "GB/s", "n_gpus": ws,
                          "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": round(sum(times) / len(times) * 1e3, 2), "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "bytes", "data": "synthetic",
                          "config": {"workload": "swap_blocks", "description": CONFIG_TEXT["swap_blocks"],
                                     "step": "48 blocks out and in on the host (bounded sample)"},
                          "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                                           "sample": "48 blocks out and in per step"},
                          "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return
    wl = _iterations(args.config, args.seed)[0]
    dtype = CONFIG_DTYPE.get(args.config, "fp16")
    threads = len(os.sched_getaffinity(0))
    oracle.set_num_threads(threads)
    samples = [_layer_sample(wl, l, None, seed=1, dtype=dtype) for l in range(2)]
    times = []
    for i in range(args.warmup + args.steps):
        mini, tables, q, n = samples[i % len(samples)]
        t0 = time.perf_counter()
        _oracle_layer(oracle, wl, mini, tables, q, n, dtype)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    if wl.num_decode:
        metric = "decode KV GB/s (KV bytes read per 32-layer iteration / iteration time) at batch 32"
        value, unit = kv_bytes(wl, len(times), dtype) / total / 1e9, "GB/s"
    else:
        metric = "prefill attention TFLOP/s"
        value, unit = 4 * HEAD_DIM * wl.q_heads * prefill_pairs(wl) * len(times) / total / 1e12, "TFLOP/s"
    res = {"impl": "reference", "metric": metric, "value": round(value, 4), "unit": unit, "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / len(times) * 1e3, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
           "data": "synthetic",
           "config": {"workload": args.config, "description": CONFIG_TEXT[args.config],
                      "step": "one layer of the first iteration (bounded sample)"},
           "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": threads, "kind": "oracle",
                            "sample": "all rows and heads of one layer per step"},
           "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="average_decode",
                    choices=["average_decode", "long_decode", "shared_prefix_decode", "mixed_prefill", "gqa_decode",
                             "average_decode_int8", "mixed_prefill_int8", "mixed_prefill_gqa", "swap_blocks",
                             "shared_prefix_cascade", "shared_prefix_cascade_gqa", "shared_prefix_cascade_int8"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch each step directly instead of replaying a CUDA graph")
    ap.add_argument("--no-prefill-schedule", action="store_true",
                    help="average_decode: skip the extra prefill-kernel timing over the 8-chunk schedule")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--seed", type=int, default=0, help="seed of the workload's length and block draws")
    ap.add_argument("--partition-tokens", type=int, default=0,
                    help="decode split-K partition size of the pool (0 = the library default)")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only this many layers (smaller pool; per-layer work unchanged; for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.config == "swap_blocks":
        run_swap(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
