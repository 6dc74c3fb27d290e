"""The N > 1 host path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The decode shards into independent (sequence, KV head) units, so ranks only
meet at a barrier and at the MAX over their step times.  Under KV-head
sharding (the default) each rank owns half of the KV heads of every
sequence and the ranks' output slices reassemble into the full output;
under replicas each rank draws its own sequences; the reference arm runs
on rank 0 alone."""
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


def test_job_throughput():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_tokens_per_s(256, 10, 1, 20.0)
    assert bench.job_tokens_per_s(256, 10, 2, 20.0) == pytest.approx(2 * one)            # replicas: weak
    assert bench.job_tokens_per_s(256, 10, 2, 10.0, "heads") == pytest.approx(2 * one)   # heads: same tokens, half the time
    assert bench.reduce_max_ms(3.0) == 3.0           # no process group: unchanged


def _oracle_rank_output(w, rank, world):
    """The decode output slice [B][H_q/N][D] of `rank` under KV-head
    sharding, computed by the oracle from the rank's own inputs: its KV
    heads' contexts (generated for those heads only), its query heads."""
    import numpy as np
    import torch
    import oracle as O
    from bit_kv_cache_quantize_gb300 import inputs as I
    from bit_kv_cache_quantize_gb300 import shard as S
    T = D = 128
    h0, h1 = S.head_range(rank, world, w.num_kv_heads)
    q = S.slice_heads(I.queries(w), rank, world, w.num_q_heads, axis=1)
    bits = lambda x: x.contiguous().view(torch.int16).numpy().view(np.uint16)
    out = np.zeros((w.batch, q.shape[1], D))
    for b in range(w.batch):
        n = w.seq_lens[b]
        k = I.kv_sequence(w, "k", b, n, heads=range(h0, h1))
        v = I.kv_sequence(w, "v", b, n, heads=range(h0, h1))
        nf = n // T
        for i in range(h1 - h0):
            kx = O.decode16(bits(k[:, i]), w.dtype)
            vx = O.decode16(bits(v[:, i]), w.dtype)
            kr = [O.pack_record(False, O.quantize_tile(kx[t * T:(t + 1) * T], 15)) for t in range(nf)]
            vr = [O.pack_record(True, O.quantize_tile(vx[t * T:(t + 1) * T], 3), v_bits=2) for t in range(nf)]
            qx = O.decode16(bits(q[b, i * w.G:(i + 1) * w.G]), w.dtype)
            out[b, i * w.G:(i + 1) * w.G] = O.attention_folded(qx, kr, vr, kx[nf * T:], vx[nf * T:], w.scale)
    return out


def _shard_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        from bit_kv_cache_quantize_gb300 import inputs as I
        w = I.Workload("shard_mix", 3, 8, 4, "f16", [300, 129, 77], seed=31, max_tokens=300, block_perm=True)
        mine = torch.from_numpy(_oracle_rank_output(w, rank, world))
        parts = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(parts, mine)               # test-side check only: the decode itself exchanges nothing
        q.put((rank, [p.numpy() for p in parts] if rank == 0 else None))
    finally:
        dist.destroy_process_group()


def test_kv_head_shards_reassemble_the_full_output():
    """Two gloo ranks each decode (oracle) their half of the KV heads from
    their own inputs; their output slices, concatenated in rank order along
    the query-head axis, equal the unsharded output index for index."""
    import numpy as np
    sys.path.insert(0, ROOT)
    from bit_kv_cache_quantize_gb300 import inputs as I
    from bit_kv_cache_quantize_gb300 import shard as S
    ctx = multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=300) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = I.Workload("shard_mix", 3, 8, 4, "f16", [300, 129, 77], seed=31, max_tokens=300, block_perm=True)
    full = _oracle_rank_output(w, 0, 1)           # one rank holding every head
    assert S.head_range(0, 2, 4) == (0, 2) and S.head_range(1, 2, 4) == (2, 4)
    assert S.q_head_range(1, 2, 4, 8) == (4, 8)
    assembled = S.assemble(got[0], axis=1)
    assert assembled.shape == full.shape == (3, 8, 128)
    assert np.array_equal(assembled, full)
    with pytest.raises(ValueError):
        S.head_range(0, 3, 8)                      # heads must divide evenly
