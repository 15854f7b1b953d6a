"""The N > 1 path of the benchmark is replicas only (the projections shard by
token rows with no exchange): each rank runs its own batch, and the job's
time is the slowest rank's.  Its host logic runs here as two gloo ranks on
the CPU: distinct per-rank inputs with shared weights, the max-over-ranks
reduction of the timed seconds, and the whole-job throughput."""
import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    import clef_synth as S
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = S.workload("int8-linear-m298-2048x2048")
        acts, weights, _ = S.layer_inputs(cfg, seed=0)
        mine = bench.replica_activations(cfg, acts, rank)
        seconds = 1.0 + rank           # rank 1 is the slow one
        tmax = bench.max_over_ranks(seconds, world, dist, "cpu")
        dist.barrier()
        out[rank] = (float(np.asarray(mine["x"], np.float64).sum()),
                     float(np.asarray(weights["proj"][0], np.float64).sum()), tmax,
                     bench.whole_job_tops(1e12, 10, world, tmax))
    finally:
        dist.destroy_process_group()


def test_two_replicas_on_gloo():
    world = 2
    port = _free_port()
    # every process of the test is spawned (the Manager's too): a fork after
    # the GPU tests of the same session have started threads could deadlock
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    (x0, w0, t0, v0), (x1, w1, t1, v1) = res[0], res[1]
    assert x0 != x1, "each replica gets its own activations"
    assert w0 == w1, "replicas share the weights"
    assert t0 == t1 == 2.0, "both ranks see the slowest rank's time"
    assert v0 == v1 == 1e12 * 10 * 2 / 2.0 / 1e12


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    import clef_synth as S
    cfg = S.workload("int8-linear-m298-2048x2048")
    acts, _, _ = S.layer_inputs(cfg, seed=0)
    assert bench.replica_activations(cfg, acts, 0) is acts
    assert bench.max_over_ranks(1.5, 1, None, "cpu") == 1.5
