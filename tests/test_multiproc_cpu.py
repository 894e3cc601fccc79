"""The bench's multi-process (N > 1) host logic, on CPU with the gloo backend.

On N GPUs every rank runs its own batch of the workload (weak scaling, no
collective on the data path).  What crosses ranks is only the step time: the
slowest rank sets the job's pace, and the job's throughput counts the tokens
of every rank.  These tests run that aggregation with two real processes
(world size 2, gloo, rendezvous on 127.0.0.1), check that the ranks draw
different batches, and that the reference arm does its work on rank 0 only.
"""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, world, port, ms_local, tokens, out):
    import torch
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench
    from hybrid_attention_ssm_fwd_b300 import synth

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_max, value = bench.job_throughput(ms_local[rank], tokens, world, torch.device("cpu"))
        s = synth._shape(B=1, T=8, M=0, d=16, Hq=2, Hkv=1, dh=8, di=32, N=4, k=4, window=0, dtype="bf16")
        x = synth.make_layer_inputs(s, bench.rank_seed(rank))["X"]
        xs = [None] * world
        dist.all_gather_object(xs, x)
        # distinct batches: every rank's input differs from every other rank's
        distinct = all(not np.array_equal(xs[i], xs[j]) for i in range(world) for j in range(i + 1, world))
        out.put((rank, ms_max, value, distinct))
    finally:
        dist.destroy_process_group()


def test_job_throughput_single_process():
    import bench
    ms, v = bench.job_throughput(2.5, 1000, 1, None)
    assert ms == 2.5 and v == pytest.approx(1000 / 2.5e-3)


def test_two_rank_gloo_max_over_ranks_and_aggregate():
    world, tokens = 2, 65536
    ms_local = [3.25, 4.5]       # rank 1 is the slower one
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, ms_local, tokens, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms_max, value, distinct in sorted(res):
        assert ms_max == max(ms_local), f"rank {rank} took {ms_max}"
        assert value == pytest.approx(tokens * world / (max(ms_local) / 1e3), rel=1e-12)
        assert distinct


@pytest.mark.parametrize("rank,expect_line", [(1, False), (0, True)])
def test_reference_arm_runs_on_rank0_only(rank, expect_line):
    env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3", "--ref-sample-tokens", "16"],
                       capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    if not expect_line:
        assert lines == []
    else:
        import json
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_bench_gpus_2_launches_two_ranks():
    """`python bench.py --gpus 2` without torchrun around it starts two ranks
    itself (torch.distributed.run on 127.0.0.1); with the CPU dry run they
    meet over gloo, and rank 0 prints one line with n_gpus 2 and the slower
    rank's step time."""
    import json
    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--dry-run-cpu",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True, timeout=240, env=env,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["n_gpus"] == 2
    assert out["ms_per_step"] == 11.0                     # ranks report 10 + rank ms
    assert out["value"] == pytest.approx(2 * 8 * 8192 / 11e-3, rel=1e-6)
