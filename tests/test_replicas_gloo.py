"""The N > 1 host logic of the benchmark, on CPU: two gloo ranks in separate processes.

Replicas exchange nothing on the data path; what crosses ranks is the slowest rank's step
time.  Checks: every rank receives the maximum, the whole-job rate counts every rank's bytes
over that time, replicas draw different data of identical shape and lengths, and the CPU
reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from kv_cache_decode_kvc_gb300 import replicas, synth
from kv_cache_decode_kvc_gb300.workloads import HEADLINE, WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, local, n = replicas.env_rank()
        assert (r, local, n) == (rank, rank, world)
        ms_local = [2.5, 3.25][rank]
        ms = replicas.max_over_ranks(ms_local, world)
        rate = replicas.whole_job_rate(world, 1.0e9, ms)
        w = WORKLOADS[HEADLINE]
        seed = replicas.replica_seed(w.seed, rank)
        q = synth.queries(seed, 0, 2, w.H_q, w.D)
        # gather every rank's first query row to rank 0 (test-only exchange)
        rows = [torch.empty_like(q[0, 0].float()) for _ in range(world)]
        dist.all_gather(rows, q[0, 0].float())
        dist.barrier()
        if rank == 0:
            torch.save({"ms": ms, "rate": rate, "rows": rows, "lens": w.lens()}, out_path)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_draw_distinct_data(tmp_path):
    out = str(tmp_path / "rank0.pt")
    mp.spawn(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True)
    got = torch.load(out)
    assert got["ms"] == 3.25                                   # the maximum, on every rank
    assert abs(got["rate"] - 2 * 1.0e9 / 3.25e-3 / 1e9) < 1e-9  # both ranks' bytes / slowest time
    a, b = got["rows"]
    assert a.shape == b.shape and not torch.equal(a, b)        # distinct replica data
    assert torch.equal(got["lens"], WORKLOADS[HEADLINE].lens())  # equal work per rank


def test_single_process_needs_no_process_group():
    assert replicas.max_over_ranks(1.5, 1) == 1.5
    assert replicas.replica_seed(1234, 0) == 1234
    assert len({replicas.replica_seed(1234, r) for r in range(8)}) == 8


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""
