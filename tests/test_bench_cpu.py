"""Host-side logic of bench.py: the byte model, the multi-rank aggregation
(world size 2 over gloo on the CPU), and the reference arm's JSON line."""

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_byte_model_serving_workload():
    w = W.make_config(3)
    # S0 64 MiB + q,k 32 MiB + v 32 MiB + gates 1 MiB + parent + o 32 MiB + U 64 MiB
    assert bench.verify_bytes(w) == 235945984
    L = int(w.path_len.sum())
    assert bench.commit_bytes(w) == (2 * 64 * 2**20 + L * 32 * 512 + L * 16 * 256
                                     + L * 32 * 4 + 32 * 25 * 4)
    assert bench.verify_kernel_name(w) == "verify_tc_kernel"
    assert bench.verify_kernel_name(W.make_config(0)) == "verify_generic_kernel"
    # the commit: CUDA cores for paths of up to 32 entries, tensor cores past them
    assert bench.commit_kernel_name(w) == "commit_kernel"
    w4 = W.make_config(4)
    assert bench.commit_kernel_name(w4) == "commit_tc_kernel"
    assert bench.verify_kernel_name(w4) == "verify_mid_kernel"
    wl = W.make_custom(seed=1, B=1, N=300, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                       tree="random", max_depth=24)
    assert bench.verify_kernel_name(wl) == "verify_chain_kernel + verify_long_tc_kernel"
    wf = W.make_custom(seed=1, B=1, N=300, Hqk=1, Hv=2, dk=64, dv=64, dtype=W.F32,
                       tree="random", max_depth=24)
    assert bench.verify_kernel_name(wf) == "verify_long_kernel"
    assert bench.topw_kernel_name(128, 4, 4) == "tree_topw_list_kernel"
    assert bench.topw_kernel_name(256, 8, 4) == "tree_topw_list_kernel"
    assert bench.topw_kernel_name(256, 8, 8) == "tree_topw_kernel"


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [2.0, 3.0][rank]  # rank 1 is the slow one
    m = bench.max_over_ranks(ms, dist)
    out[rank] = (m, bench.job_throughput(world, 32, 128, m))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_over_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = 29500 + os.getpid() % 1000
    ps = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 3.0
    assert out[0][1] == pytest.approx(2 * 32 * 128 / 3e-3)


def _small(cfg, seed):
    return W.make_custom(seed=seed, B=2, N=12, Hqk=1, Hv=2, dk=16, dv=16, dtype=W.F32,
                         tree="mixed")


def _shard_rank(rank, world, port, out):
    import numpy as np
    import torch
    import torch.distributed as dist
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = bench.rank_workload(3, rank, make=_small)
    o, U = oracle.verify_workload(w, threads=1)
    S1 = oracle.commit_workload(w, threads=1)
    got = {k: bench.gather_sequences(torch.from_numpy(np.ascontiguousarray(a)), dist, world)
           for k, a in (("o", o), ("U", U), ("S1", S1))}
    out[rank] = {k: v.numpy() for k, v in got.items()}
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_batches_reassemble_to_the_job():
    """Each rank verifies its own seeded batch; gathered in rank order, the
    per-sequence results equal the job computed in one process over the
    concatenated batches (rank r's sequences at index r * B)."""
    import numpy as np
    import oracle
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = 29700 + os.getpid() % 1000
    ps = [ctx.Process(target=_shard_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    ws = [bench.rank_workload(3, r, make=_small) for r in range(2)]
    assert not np.array_equal(ws[0].q, ws[1].q)  # independent batches
    for r in range(2):
        o, U = oracle.verify_workload(ws[r], threads=1)
        S1 = oracle.commit_workload(ws[r], threads=1)
        for k, a in (("o", o), ("U", U), ("S1", S1)):
            for rank in range(2):
                np.testing.assert_array_equal(out[rank][k][r * 2:(r + 1) * 2], a)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "nodes/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    # the whole layer is timed every step, with the same workload keys as our arm
    assert "whole layer" in d["cpu_baseline"]["sample"]
    w = W.make_config(3)
    assert d["config"] == bench.workload_config(w, 1)
