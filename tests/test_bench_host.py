"""Host-side logic of bench.py: algorithmic work counts, clock summaries, and
the cross-rank timing aggregation run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
import seeded_inputs as si


def test_live_pair_counts():
    # causal keeps i+1 keys per row; with a window min(i+1, W); bidirectional S keys
    assert bench.live_pairs(5, True, 0) == 15
    assert bench.live_pairs(5, False, 0) == 25
    assert bench.live_pairs(4096, True, 1024) == 3670528
    assert bench.live_pairs(6, False, 2) == 6 + 2 * 5


def test_workload_work_figures():
    # vision: 4 * S^2 * D * H
    class C:
        seq_len, head_dim, n_heads, causal, window = 2304, 64, 16, False, 0
    assert bench.prefill_flops(C) == 4 * 2304 * 2304 * 64 * 16
    tiny = si.make_workload("tiny_decode")
    # 128 tokens * 2 kv heads * 64 dims * 2 bytes * (K + V) + q + out + kv_len
    assert bench.decode_bytes(tiny) == 128 * 2 * 64 * 2 * 2 + 2 * 4 * 64 * 2 + 4


def test_chunk_ring_tiered_and_f32_work_figures():
    # chunked prefill: a chunk of n queries at the end of L keys keeps pos + 1 keys
    # for query pos = L - n + i (none below position 0)
    class Ch:
        q_lens, kv_lens, window, head_dim, n_heads = [3, 2], [5, 1], 0, 8, 2
    pairs = (3 + 4 + 5) + (1)   # sequence 0: positions 2,3,4; sequence 1: position 0 (and -1)
    assert bench.chunk_flops(Ch) == 4 * 8 * pairs * 2
    # ring: a 16-slot ring keeps min(L, 16) tokens whatever the logical length
    c = si.make_decode_case(2, 4, 2, 16, [40, 7], seed=1, ring=16)
    per_tok = 2 * 16 * 2 * 2
    assert bench.decode_bytes(c) == (16 + 7) * per_tok + 2 * 4 * 16 * 2 + 2 * 4 * 16 * 2 + 2 * 4
    # f32 queries and outputs: 4 bytes each instead of 2
    c32 = si.make_decode_case(2, 4, 2, 16, [40, 7], seed=1, ring=16, q_f32=True)
    assert bench.decode_bytes(c32, 4) == (16 + 7) * per_tok + 2 * 4 * 16 * 4 * 2 + 2 * 4
    # tiered: kept cold tokens (int8 codes + 2 f16 scales per kv head) and kept hot ring tokens
    t = si.make_tiered_case(2, 4, 2, 16, [10, 3], [20, 5], 16, seed=2, int8=True, window=12)
    cold_tok = 2 * 16 * 2 + 2 * 2 * 2
    hot_tok = 2 * 16 * 2 * 2
    # window 12: sequence 0 keeps 12 hot tokens (of the 16 the ring holds) and no cold
    # one; sequence 1 keeps its 5 hot tokens and min(3, 12 - 5) = 3 cold ones
    kv = (0 * cold_tok + 12 * hot_tok) + (3 * cold_tok + 5 * hot_tok)
    assert bench.tiered_bytes(t) == kv + 2 * 4 * 16 * (2 + 2) + 3 * 2 * 4


def test_clock_summary_flags_throttle_reasons():
    lines = ["0, 1900, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active",
             "0, 1950, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1920, 2070, 940.0, 0x0, Active, Not Active, Not Active, Not Active"]
    s = bench.ClockSampler.summary(lines)
    assert s["sm_mhz"] == 1920 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(1.0 + rank, world)
    s = bench.sum_over_ranks(10.0 * (rank + 1), world)
    bench.barrier(world)
    q.put((rank, t, s))
    dist.destroy_process_group()


def test_two_rank_timing_aggregation_gloo():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2.0, 30.0), (1, 2.0, 30.0)]
