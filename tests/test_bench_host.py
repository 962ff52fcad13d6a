"""Host-side logic of bench.py: the multi-rank timing reduction over a
world-size-2 gloo process group on CPU, the whole-job throughput, the clock
record parser, and the algorithmic work counts the roofline uses."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 10 + r ms for the step and 5 - r ms end to end
        got = bench.max_over_ranks([10.0 + rank, 5.0 - rank], dist)
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_timing_reduction_takes_the_slowest_rank_on_every_rank():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    assert dict(out) == {0: [11.0, 5.0], 1: [11.0, 5.0]}


def test_whole_job_throughput_is_all_work_over_the_slowest_rank():
    assert bench.aggregate([10.0, 11.0], [100, 100]) == pytest.approx(200 / 0.011)
    assert bench.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]


def test_clock_record_parsing():
    lines = ["2070, 2070, 240.1, 0x0, Not Active, Not Active, Not Active, Not Active",
             "1900, 2070, 900.5, 0x4, Not Active, Not Active, Not Active, Active",
             "2070, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    c = bench.parse_clock_lines(lines)
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070 and c["reasons"] == ["sw_power_cap"]
    assert c["samples"] == 3 and c["power_w_max"] == 900.5


def test_algorithmic_work_counts():
    # 13 rows x 8,192 tokens x 16,384 B per token and layer x 32 layers = 55.83 GB
    assert bench.kv_bytes(workloads.long_decode(0), 32) == 55834574848
    # one 4,000-token prompt: sum over positions p of (p + 1) pairs = 8,002,000
    pairs = sum(bench.prefill_pairs(workloads.mixed_prefill(c)) for c in range(8))
    assert pairs == 4000 * 4001 // 2
    # chunk 6 covers positions 3,072..3,583
    assert bench.prefill_pairs(workloads.mixed_prefill(6)) == 1704192


def test_every_workload_fits_the_pool_and_tables_are_disjoint():
    for wl in [workloads.tiny_decode(0), workloads.average_decode(0), workloads.long_decode(0),
               workloads.mixed_prefill(7)]:
        used = wl.block_tables[wl.block_tables >= 0]
        assert len(np.unique(used)) == len(used) and used.max() < wl.num_blocks
        for r in range(wl.num_seqs):
            assert (wl.block_tables[r] >= 0).sum() * 16 >= wl.ctx_lens[r]
    sp = workloads.shared_prefix_decode(0)
    assert (sp.block_tables[:, :125] == sp.block_tables[0, :125]).all()
    assert ((sp.ctx_lens >= 2001) & (sp.ctx_lens <= 2300)).all()


def test_prefill_chunk_roofline_splits_hbm_and_tensor_bound_chunks():
    # the 4,000-token prompt's 8 chunks at the same time each: the first two chunks' FLOPs per byte sit below
    # the ridge (1,946.2 TFLOP/s over 6,783.5 GB/s = 287 FLOP/B), the rest above it
    its = [workloads.mixed_prefill(c) for c in range(8)]
    r = bench.prefill_chunk_summary([(w, 20.0, 32, 32, 256) for w in its], 6783.5, 1946.2, "measured")
    assert [c["bound"] for c in r["per_chunk"]] == ["hbm"] * 2 + ["tensor"] * 6
    # chunk c (c < 7) has 512 queries at positions 512c .. 512c + 511: 512 x 512c + 512 x 513 / 2 pairs;
    # chunk 7 has 416 queries at 3,584 .. 3,999
    pairs = [512 * 512 * c + 512 * 513 // 2 for c in range(7)] + [416 * 3584 + 416 * 417 // 2]
    flops = [4 * 128 * 32 * p for p in pairs]
    assert r["aggregate"]["tflops"] == pytest.approx(sum(flops) / (8 * 20e-6) / 1e12, abs=0.1)
    assert r["aggregate_tensor_bound"]["chunks"] == 6
    assert r["aggregate_tensor_bound"]["tflops"] == pytest.approx(sum(flops[2:]) / (6 * 20e-6) / 1e12, abs=0.1)


def test_kernel_source_hash_ignores_comments_but_not_code():
    a = "int f(int x) {\n    // the sum\n    return x + 1;  /* one */\n}\n"
    b = "int f(int x) {\n\n    return x + 1;\n}\n/* a longer\n   comment */\n"
    c = "int f(int x) {\n    return x + 2;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
