"""Benchmark: one engine iteration (32 layers) of paged decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: for every one of the
32 layers, kv_append of each row's new token and decode attention of every
row over its paged context, through libpkv's C ABI (pkv_step). Default
workload: batch-32 decode with prompt lengths from a clipped lognormal (mean
1,250, 50..8,000) plus U{0..299} generated tokens, over a 7,152-block (60 GB)
pool with shuffled block ids, N(0,1) FP16 values (synthetic; no dataset).

One JSON line is printed by rank 0. Under torchrun (N > 1) every rank runs
its own replica of the workload (weak scaling, no collective on the data
path); `value` adds the KV bytes of all ranks over the slowest rank's time.

`--impl reference` times the oracle (plain CPU code, oracle/) on the host
cores on a bounded sample of the same workload: one layer per step.
"""
from __future__ import annotations

import argparse
import hashlib
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

KV_BYTES_PER_TOKEN_LAYER = 2 * 32 * 128 * 2          # K and V of 32 heads x 128 dims, FP16: 16,384 B
SCALE = float(np.float32(1.0 / np.sqrt(np.float32(128.0))))

CONFIGS = {
    "average_decode": lambda: workloads.average_decode(0),
    "long_decode": lambda: workloads.long_decode(0),
    "shared_prefix_decode": lambda: workloads.shared_prefix_decode(0),
}
CONFIG_TEXT = {
    "average_decode": "batch-32 decode, 32 layers x 32 heads x 128 fp16, context = clipped lognormal prompt "
                      "(mean 1,250) + U{0..299} generated + 1, 7,152-block (60 GB) shuffled pool, kv_append of 1 "
                      "token per row",
    "long_decode": "13 rows x 8,192 context tokens, 32 layers, 7,152-block pool, split-K partitions",
    "shared_prefix_decode": "64 rows sharing 125 ref-counted prefix blocks + 1..300 private tokens, 32 layers",
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


KERNEL_SOURCES = {
    "decode_attn": ["pkv_kernels.cu", "ptx.cuh", "pkv_internal.h"],
    "prefill_attn": ["pkv_prefill.cu", "ptx.cuh", "pkv_internal.h"],
}


def _kernel_source_hash(kernel: str):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_scatter_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
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
                                          "--format=csv,noheader,nounits", "-lms", "200"],
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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


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


# ------------------------------------------------------------------ ours

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

    wl = CONFIGS[args.config]()
    if args.layers:
        wl.num_layers = args.layers          # same per-layer work, fewer layers (profiling runs)
    L, H, D = wl.num_layers, wl.num_heads, wl.head_dim
    B, T, S = wl.num_seqs, wl.num_tokens, wl.num_seqs
    dev = torch.device("cuda", local)

    pool_t = torch.empty(workloads.pool_shape(wl.num_blocks, L, H), dtype=torch.float16, device=dev)
    workloads.fill_normal_fp16_(pool_t, workloads.value_seed(wl.seed, "pool"))
    pool = pkv.Pool(pool_t, wl.num_blocks, num_layers=L, num_heads=H)

    tables, ctx, slots, qs = _metadata_via_block_manager(pkv, pool, wl)
    tables_h = torch.from_numpy(tables).pin_memory()
    ctx_h = torch.from_numpy(ctx).pin_memory()
    qs_h = torch.from_numpy(qs).pin_memory()
    slots_h = torch.from_numpy(slots).pin_memory()
    tables_d, ctx_d, qs_d, slots_d = (x.to(dev) for x in (tables_h, ctx_h, qs_h, slots_h))

    gen = torch.Generator(device=dev)
    gen.manual_seed(workloads.value_seed(wl.seed, "q"))
    q = torch.randn((L, T, H, D), generator=gen, device=dev).half()
    k = torch.randn((L, T, H, D), generator=gen, device=dev).half()
    v = torch.randn((L, T, H, D), generator=gen, device=dev).half()
    out = torch.empty_like(q)
    stride = T * H * D
    desc = pkv.make_step_desc(num_decode=B, num_prefill=0, num_tokens=T, max_q_len=0, max_blocks=wl.max_blocks,
                              first_layer=0, num_layers=L, scale=SCALE, block_tables=tables_d, ctx_lens=ctx_d,
                              q_start_loc=qs_d, slot_mapping=slots_d, q=q, k=k, v=v, out=out,
                              q_layer_stride=stride, k_layer_stride=stride, v_layer_stride=stride,
                              out_layer_stride=stride)
    wsb = pool.step_workspace_bytes(desc)
    wspace = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        pool.step(desc, wspace, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st, flags = pool.get_status(stream)
    if st != pkv.PKV_OK:
        raise RuntimeError(f"device status {st} flags {flags:#x}")

    kv_bytes_step = int(wl.ctx_lens.astype(np.int64).sum()) * KV_BYTES_PER_TOKEN_LAYER * L
    att_tokens_step = int(wl.ctx_lens.astype(np.int64).sum())
    max_parts = -(-wl.max_blocks * 16 // 512)
    launches_per_layer = 2 + (1 if max_parts > 1 else 0)

    sampler = ClockSampler(_gpu_id(torch, local))
    # ---- timed region 1: the whole step through pkv_step
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    t_ms = e0.elapsed_time(e1)

    # ---- timed region 2: same work layer by layer, events around every decode call
    dec_ev = []
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e2.record(stream)
    for _ in range(args.steps):
        for l in range(L):
            pool.kv_append(l, k[l], v[l], slots_d, stream)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            pool.decode_attn(l, q[l], tables_d, ctx_d, SCALE, out[l], wspace, stream)
            b.record(stream)
            dec_ev.append((a, b))
    e3.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    t2_ms = e2.elapsed_time(e3)
    dec_ms = [a.elapsed_time(b) for a, b in dec_ev]
    dec_avg_ms = sum(dec_ms) / len(dec_ms)

    # ---- end to end: host buffers in, host result out, every step
    q_h, k_h, v_h = (x.cpu().pin_memory() for x in (q, k, v))
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e4, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e4.record(stream)
    for _ in range(args.steps):
        for src, dst in ((q_h, q), (k_h, k), (v_h, v), (tables_h, tables_d), (ctx_h, ctx_d), (qs_h, qs_d),
                         (slots_h, slots_d)):
            dst.copy_(src, non_blocking=True)
        step()
        out_h.copy_(out, non_blocking=True)
    e5.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e4.elapsed_time(e5)
    h2d = sum(x.numel() * x.element_size() for x in (q_h, k_h, v_h, tables_h, ctx_h, qs_h, slots_h))
    d2h = out_h.numel() * out_h.element_size()
    st, flags = pool.get_status(stream)
    if st != pkv.PKV_OK:
        raise RuntimeError(f"device status {st} flags {flags:#x}")

    # max over ranks
    times = torch.tensor([t_ms, e2e_ms, dec_avg_ms], dtype=torch.float64, device=dev)
    if ws > 1:
        dist.all_reduce(times, op=dist.ReduceOp.MAX)
    t_ms, e2e_ms, dec_avg_ms = (float(x) for x in times.tolist())

    hbm_peak, tf_peak, peak_kind = _peaks()
    total_kv = kv_bytes_step * args.steps * ws
    value = total_kv / (t_ms * 1e-3) / 1e9
    dec_bytes = int(wl.ctx_lens.astype(np.int64).sum()) * KV_BYTES_PER_TOKEN_LAYER + 2 * B * H * D * 2
    achieved = dec_bytes / (dec_avg_ms * 1e-3) / 1e9
    traffic = _traffic("decode_attn", args.config)

    result = {
        "metric": "decode KV GB/s (KV bytes read per 32-layer iteration / iteration time) at batch 32",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_ms / args.steps, 4),
        "us_per_iteration": round(t_ms / args.steps * 1e3, 1),
        "attention_tokens_per_s": round(att_tokens_step * L * args.steps * ws / (t_ms * 1e-3), 1),
        "hbm_frac_of_measured_peak": round(value / hbm_peak, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 storage, f32 arithmetic",
        "data": "synthetic",
        "config": {"workload": args.config, "description": CONFIG_TEXT[args.config], "num_layers": L,
                   "num_seqs": B, "heads": H, "head_dim": D, "pool_blocks": wl.num_blocks,
                   "context_tokens": att_tokens_step, "max_context": int(wl.ctx_lens.max()),
                   "kv_bytes_per_step": kv_bytes_step, "seed": wl.seed,
                   "l2": "inputs larger than L2 (every step reads the whole KV context of all 32 layers)"},
        "clocks": clocks,
        "gpu_launches": launches_per_layer * L * args.steps,
        "roofline": {"bound": "hbm", "kernel": "decode_attn (decode_kernel + reduce_kernel)",
                     "achieved": round(achieved, 1), "peak": hbm_peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": dec_bytes, "avg_launch_us": round(dec_avg_ms * 1e3, 2),
                     "layerwise_ms_per_step": round(t2_ms / args.steps, 4)},
        "e2e": {"value": round(total_kv / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms / args.steps, 4)},
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl, pool_t, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def _metadata_via_block_manager(pkv, pool, wl):
    """Step metadata from libpkv's block manager, as a serving loop would get it.

    The pool hands blocks out in the workload's permutation order, so the
    tables equal the workload's own (checked)."""
    nb_used = int(np.unique(wl.block_tables[wl.block_tables >= 0]).size)
    perm = np.concatenate([wl.block_tables[r][wl.block_tables[r] >= 0] for r in range(wl.num_seqs)])
    _, first = np.unique(perm, return_index=True)
    order = perm[np.sort(first)]
    rest = np.setdiff1d(np.arange(wl.num_blocks), order)
    pool_order = np.concatenate([order, rest]).astype(np.int64)
    mgr = pkv.Pool(None, wl.num_blocks, num_layers=wl.num_layers, num_heads=wl.num_heads, free_order=pool_order)
    prefix = int(wl.meta.get("prefix_blocks", 0))
    if prefix:
        assert mgr.seq_grow(-1, prefix * 16) == pkv.PKV_OK
    for r in range(wl.num_seqs):
        if prefix:
            assert mgr.seq_share_prefix(r, -1, prefix) == pkv.PKV_OK
        assert mgr.seq_grow(r, int(wl.ctx_lens[r])) == pkv.PKV_OK
    st, tables, ctx, slots, qs = mgr.build_step(np.arange(wl.num_seqs), wl.q_lens, wl.max_blocks)
    assert st == pkv.PKV_OK and np.array_equal(tables, wl.block_tables) and np.array_equal(ctx, wl.ctx_lens)
    assert mgr.free_blocks() == wl.num_blocks - nb_used
    return tables, ctx, slots, qs


# ------------------------------------------------------------------ oracle timings

def _layer_sample(wl, layer, pool_t=None, seed=0):
    """Host mini-pool of one layer's referenced blocks (renumbered), its tables and q."""
    import torch
    nb = -(-wl.ctx_lens.astype(np.int64) // 16)
    ids = np.concatenate([wl.block_tables[r, :nb[r]] for r in range(wl.num_seqs)]).astype(np.int64)
    uniq, inv = np.unique(ids, return_inverse=True)
    if pool_t is not None:
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
    q = workloads.normal_fp16((wl.num_seqs, wl.num_heads, 128), workloads.value_seed(wl.seed, "q", layer)).numpy()
    return np.ascontiguousarray(mini), tables, q.view(np.uint16), len(uniq)


def cpu_baseline(wl, pool_t, budget_s):
    import oracle
    threads = len(os.sched_getaffinity(0))
    oracle.set_num_threads(threads)
    done_bytes, t_total, layers = 0, 0.0, 0
    for layer in range(wl.num_layers):
        mini, tables, q, n = _layer_sample(wl, layer, pool_t)
        g = oracle.geom(n, 1, wl.num_heads)
        t0 = time.perf_counter()
        oracle.decode_attn(mini, g, 0, q, tables, wl.ctx_lens, SCALE)
        t_total += time.perf_counter() - t0
        done_bytes += int(wl.ctx_lens.astype(np.int64).sum()) * KV_BYTES_PER_TOKEN_LAYER
        layers += 1
        if t_total >= budget_s:
            break
    return {"value": round(done_bytes / t_total / 1e9, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"decode attention of all {wl.num_seqs} rows x {wl.num_heads} heads for {layers} of "
                      f"{wl.num_layers} layers (referenced blocks copied to host first, copy not timed)",
            "seconds": round(t_total, 2)}


def run_reference(args):
    ws, rank, local = _dist()
    if rank != 0:
        return
    import oracle
    wl = CONFIGS[args.config]()
    threads = len(os.sched_getaffinity(0))
    oracle.set_num_threads(threads)
    samples = [_layer_sample(wl, l % wl.num_layers, None, seed=1) for l in range(min(2, wl.num_layers))]
    per_step = int(wl.ctx_lens.astype(np.int64).sum()) * KV_BYTES_PER_TOKEN_LAYER
    times = []
    for i in range(args.warmup + args.steps):
        mini, tables, q, n = samples[i % len(samples)]
        t0 = time.perf_counter()
        oracle.decode_attn(mini, oracle.geom(n, 1, wl.num_heads), 0, q, tables, wl.ctx_lens, SCALE)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = per_step * len(times) / total / 1e9
    res = {"impl": "reference", "metric": "decode KV GB/s (KV bytes read per 32-layer iteration / iteration time) "
                                          "at batch 32",
           "value": round(value, 3), "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(total / len(times) * 1e3, 2), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
           "config": {"workload": args.config, "description": CONFIG_TEXT[args.config],
                      "step": "one layer of the iteration (bounded sample)"},
           "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
                            "sample": "decode attention of all rows and heads of one layer per step"},
           "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="average_decode", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--layers", type=int, default=0,
                    help="run only this many layers (smaller pool; per-layer work unchanged; for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
