"""Multi-process host logic of the replica bench on CPU (gloo, world size 2).

The scoring path does not shard: at N GPUs the bench runs N independent
replicas, one process per GPU.  There is no data-path collective.  The job's
time is the slowest rank's time, and its throughput counts every rank's
tokens.  These tests run that logic as two gloo ranks on the CPU.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        r, w, _ = bench.dist_env()
        # the slowest rank sets the job time
        local_ms = 10.0 if rank == 0 else 25.0
        value, total_ms = bench.replica_throughput(w, 1000, 5, local_ms)
        mx = bench.max_over_ranks(float(rank) + 1.5, w)
        bench.barrier(w)
        q.put((r, w, value, total_ms, mx))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_job_time_and_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r for r, *_ in res] == [0, 1]
    for r, w, value, total_ms, mx in res:
        assert w == 2
        assert total_ms == 25.0                     # max over ranks, not the local time
        assert value == pytest.approx(2 * 1000 * 5 / 0.025)   # both replicas' tokens / the slowest time
        assert mx == 2.5


def test_single_process_needs_no_process_group():
    import bench
    value, total_ms = bench.replica_throughput(1, 1000, 4, 8.0)
    assert total_ms == 8.0 and value == pytest.approx(1000 * 4 / 0.008)
    assert bench.max_over_ranks(3.0, 1) == 3.0
    bench.barrier(1)


def test_kernel_digest_ignores_comments_and_whitespace():
    """The DRAM-traffic record is keyed to the scoring kernels' code: comment and
    whitespace edits leave the key unchanged, code edits (even inside string
    literals) change it."""
    import bench
    base = 'int a = 1;  // note\n/* block */ asm("x // y");\n'
    assert bench._code_only(base) == bench._code_only('int a = 1;\n\n   asm("x // y");  // other note\n')
    assert bench._code_only(base) != bench._code_only(base.replace("a = 1", "a = 2"))
    assert bench._code_only(base) != bench._code_only(base.replace("x // y", "x // z"))
