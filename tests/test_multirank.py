"""The benchmark's multi-replica plumbing on CPU: world_size-2 gloo process groups stand in for
the per-GPU ranks that torch.distributed.run launches (NCCL on the GPU machine)."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        bench.barrier(world)
        ms_max = bench.max_over_ranks(ms[rank], world)
        bench.barrier(world)
        q.put((rank, ms_max, bench.job_tokens_per_s(ms_max, world, 512, 4)))
    finally:
        dist.destroy_process_group()


def _run(world, ms):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


@pytest.mark.parametrize("world,ms", [(2, [10.0, 12.5]), (3, [7.0, 3.0, 5.0])])
def test_slowest_rank_sets_the_job_time(world, ms):
    out = _run(world, ms)
    slow = max(ms)
    assert [r for r, _, _ in out] == list(range(world))
    for _, ms_max, tok in out:
        assert ms_max == slow                      # every rank sees the slowest replica
        assert tok == pytest.approx(world * 512 * 4 / (slow / 1e3))  # tokens of all ranks


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 runs and prints the reference line; the others exit 0 silently
    (and never touch a GPU or the oracle)."""
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
