"""The multi-GPU form of the benchmark, on CPU: replicas only (every rank runs
the whole path on its own inputs, no collective on the data path).  Two
`gloo` ranks check the host-side pieces the GPU runs use: the timing barrier,
the maximum over ranks that sets the step time, per-rank input seeds, and the
whole-job throughput."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import attn_inputs as gen


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        local_ms = [3.0, 5.0][rank]  # the second replica is slower
        bench.barrier(world)
        ms = bench.allmax(world, local_ms)
        cfg = dict(gen.WORKLOADS["gqa_causal_8k"])
        seed = bench.replica_seed(cfg, rank)
        fwd, bwd = bench.flops(cfg)
        out[rank] = (ms, seed, bench.job_throughput(world, fwd + bwd, ms))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_replicas_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    (ms0, seed0, v0), (ms1, seed1, v1) = res[0], res[1]
    assert ms0 == ms1 == 5.0            # every rank times the slowest replica
    assert seed0 != seed1               # each replica draws its own inputs
    cfg = gen.WORKLOADS["gqa_causal_8k"]
    import bench
    fwd, bwd = bench.flops(cfg)
    assert v0 == v1 == pytest.approx(2 * (fwd + bwd) / 5e-3)  # whole job, slowest rank's time


def test_replica_inputs_differ():
    cfg = dict(gen.WORKLOADS["tiny_mha"])
    import bench
    a = gen.make_inputs(**dict(cfg, seed=bench.replica_seed(cfg, 0)))
    b = gen.make_inputs(**dict(cfg, seed=bench.replica_seed(cfg, 1)))
    assert not torch.equal(a["q"], b["q"])
