"""Replicas across ranks (no GPU): the timing aggregation of the N-rank bench
on two gloo ranks, and the reference arm launched by torchrun with two ranks
(rank 0 alone runs and prints its line; the other exits 0)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

from smoothquant_w8a8_int8_gb300 import replicas

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                                         rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank            # this rank's elapsed time (ms)
        replicas.barrier()
        slowest = replicas.max_over_ranks(mine)
        seeds = [replicas.rank_seed(1000 + i, rank) for i in range(3)]
        res = {"rank": rank, "slowest": slowest, "seeds": seeds,
               "tops": replicas.whole_job_tops(10 ** 12, world, slowest)}
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump(res, f)
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_aggregate(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn")
    r = [json.load(open(tmp_path / f"r{k}.json")) for k in range(world)]
    # both ranks see the slowest rank's time; the job's value counts both ranks' work
    assert r[0]["slowest"] == r[1]["slowest"] == 15.0
    assert r[0]["tops"] == r[1]["tops"] == pytest.approx(2 * 1e12 / 15e-3 / 1e12)
    # the ranks' inputs are distinct shards
    assert not set(r[0]["seeds"]) & set(r[1]["seeds"])


# Offsets the benchmark and the input recipe add to a GEMM's seed: X, the
# calibration batch, the LayerNorm parameters, W, bias and residual.
DERIVED_OFFSETS = (0, 555, 4242, 7919, 104729, 1299709)


def _seed_set(rank):
    from smoothquant_w8a8_int8_gb300 import workloads as wl
    out = set()
    for w in wl.WORKLOADS.values():
        for layer in range(w.layers):
            for idx in range(len(w.linears)):
                base = replicas.rank_seed(wl.gemm_seed(w, layer, idx), rank)
                out.update(base + o for o in DERIVED_OFFSETS)
    return out


def test_rank_seed_sets_disjoint_for_eight_ranks():
    """Every seed one rank draws from (for every workload, GEMM and derived
    stream) is drawn by no other rank, for 8 ranks."""
    sets = [_seed_set(r) for r in range(8)]
    for a in range(8):
        for b in range(a + 1, 8):
            assert not sets[a] & sets[b], (a, b)
    # the derived offsets themselves are what the recipe uses
    from smoothquant_w8a8_int8_gb300 import workloads as wl
    import inspect
    src = inspect.getsource(wl)
    for o in (7919, 104729, 1299709):
        assert f"seed + {o}" in src


def test_single_process_aggregation_is_identity():
    assert replicas.max_over_ranks(3.25) == 3.25
    assert replicas.whole_job_tops(2 * 10 ** 12, 1, 1000.0) == pytest.approx(2.0)
    replicas.barrier()  # no process group: nothing to do


def test_reference_arm_under_torchrun_two_ranks():
    import oracle
    oracle.build()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--workload", "bert_large_qkv_slice_m256",
           "--reference-step-seconds", "0.05"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
