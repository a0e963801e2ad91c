"""The multi-GPU benchmark path on CPU: two gloo ranks.

bench.py under torchrun runs one independent replica of the workload per
rank (requests shard with no collective), brackets the timed region with
barriers, takes the slowest rank's time and reports the whole job's
throughput from rank 0.  These tests run that host logic with world size 2
on the gloo backend; no GPU is involved.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        # rank r took 10 + 7 r ms; the job took as long as its slowest rank
        job_ms = bench.slowest_ms(10.0 + 7.0 * rank, world, "cpu")
        dist.barrier()
        q.put((rank, job_ms, bench.job_tokens_per_s(32, world, job_ms / 1e3)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in procs)
    assert [g[0] for g in got] == [0, 1]
    for _, job_ms, tps in got:
        assert job_ms == pytest.approx(17.0)
        # 2 ranks x 32 tokens per step / 17 ms
        assert tps == pytest.approx(2 * 32 / 0.017)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_ms(3.5, 1, "cpu") == 3.5
    assert bench.job_tokens_per_s(10, 1, 0.5) == pytest.approx(20.0)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0", "--workload", "swa_tiny", "--ref-tokens", "2"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    if rank != 0:
        assert lines == []
    else:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
        assert d["cpu_baseline"]["kind"] == "oracle"
        assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
