"""The N > 1 path of the benchmark is replicas only (the projections shard by
token rows with no exchange): each rank runs its own batch, and the job's
time is the slowest rank's.  Its host logic runs here as two gloo ranks on
the CPU: distinct per-rank inputs with shared weights, the max-over-ranks
reduction of the timed seconds, and the whole-job throughput.  The reference
arm (the oracle timed on the host cores) prints its one line on rank 0 only."""
import json
import os
import socket
import subprocess
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


def _bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_other_ranks_exit_without_work():
    p = _bench({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"},
               "--steps", "1", "--warmup", "0", "--config", "int8-linear-m298-2048x2048")
    assert p.returncode == 0 and p.stdout.strip() == ""


def test_reference_arm_prints_one_line():
    p = _bench({"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"},
               "--steps", "1", "--warmup", "0", "--config", "int8-linear-m298-2048x2048")
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["config"]["workload"] == "int8-linear-m298-2048x2048"
    assert d["value"] > 0 and d["unit"] == "TOPS" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
