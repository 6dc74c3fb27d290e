"""The N > 1 host path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The decode shards into independent (sequence, KV head) units, so ranks only
meet at a barrier and at the MAX over their step times; each rank draws its
own sequences; the reference arm runs on rank 0 alone."""
import multiprocessing
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        import bench
        from bit_kv_cache_quantize_gb300 import inputs as I
        dist.barrier()
        ms = bench.reduce_max_ms(10.0 + 5.0 * rank)
        lens = I.ragged_32b(steps=4, seed=bench.rank_seed(rank)).seq_lens

        class A:
            steps, warmup, ref_seqs = 1, 0, 1
        ref = bench.run_reference(A, rank, world) if rank != 0 else "skipped"
        q.put((rank, ms, lens[:8], ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict()
    for _ in range(2):
        rank, ms, lens, ref = q.get(timeout=120)
        got[rank] = (ms, lens, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0][0] == got[1][0] == 15.0            # both ranks report the slowest rank's time
    assert got[0][1] != got[1][1]                    # disjoint work: each rank draws its own sequences
    assert got[1][2] is None                         # the reference arm does no work off rank 0


def test_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_tokens_per_s(256, 10, 1, 20.0)
    assert bench.job_tokens_per_s(256, 10, 2, 20.0) == pytest.approx(2 * one)
    assert bench.reduce_max_ms(3.0) == 3.0           # no process group: unchanged
