"""Multi-process (world size 2, gloo, CPU) checks of the head-sharded path.

Attention heads are independent, so splitting heads over ranks must give the
same result as one rank computing all of them; the timing bookkeeping takes
the max over ranks.  The per-rank attention here is the fp64 oracle (no GPU
needed); on GPUs the ranks call the library on their own heads.
"""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from io_aware_exact_10_gb300.replicas import head_shard, max_over_ranks, whole_job_rate


def test_head_shard_partitions():
    for n in (0, 1, 5, 16, 1024, 1023):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                lo, hi = head_shard(n, world, r)
                assert 0 <= lo <= hi <= n
                seen.extend(range(lo, hi))
            assert seen == list(range(n))
    with pytest.raises(ValueError):
        head_shard(4, 2, 2)


def test_whole_job_rate():
    assert whole_job_rate(10.0, 4, 2.0) == 20.0
    with pytest.raises(ValueError):
        whole_job_rate(1.0, 1, 0.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from io_aware_exact_10_gb300 import workloads as W
    w = W.Workload("mp", 2, 3, 48, 8, causal=True, seed=9)
    q, k, v, dO = W.make_inputs(w)
    BH = w.B * w.H
    flat = lambda t: t.reshape(BH, w.N, w.d).double().numpy()
    lo, hi = head_shard(BH, world, rank)
    o, lse = oracle.attn_fwd(flat(q)[lo:hi], flat(k)[lo:hi], flat(v)[lo:hi], w.scale, True)
    dq, dk, dv = oracle.attn_bwd(flat(q)[lo:hi], flat(k)[lo:hi], flat(v)[lo:hi],
                                 flat(dO)[lo:hi], w.scale, True)
    # gather every rank's shard on rank 0 (test-only; the library path has no
    # data collective)
    parts = [None] * world
    dist.all_gather_object(parts, (lo, hi, o, lse, dq, dk, dv))
    t = max_over_ranks(1.0 + rank)
    if rank == 0:
        o_all, lse_all = oracle.attn_fwd(flat(q), flat(k), flat(v), w.scale, True)
        g_all = oracle.attn_bwd(flat(q), flat(k), flat(v), flat(dO), w.scale, True)
        ok = t == float(world)
        for lo_, hi_, o_, l_, dq_, dk_, dv_ in parts:
            ok &= np.array_equal(o_, o_all[lo_:hi_]) and np.array_equal(l_, lse_all[lo_:hi_])
            for a, b in zip((dq_, dk_, dv_), g_all):
                ok &= np.array_equal(a, b[lo_:hi_])
        ok &= sum(p[1] - p[0] for p in parts) == BH
        with open(result_path, "w") as f:
            f.write("ok" if ok else "mismatch")
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_head_sharding(tmp_path):
    world = 2
    result = str(tmp_path / "result.txt")
    mp.start_processes(_worker, args=(world, _free_port(), result), nprocs=world,
                       join=True, start_method="spawn")
    assert open(result).read() == "ok"
