"""bench.py's multi-rank host logic on CPU, as world_size-2 gloo ranks: the
rank environment, the max-over-ranks timing and the whole-job rate of N
replicas, the barrier, the shared host-pool file written once by rank 0, and
the reference arm doing no work on ranks other than 0.  (The data path has no
collective: each replica serves its own tokens.)"""
import os
import socket
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, pool_dir, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), FT_POOL_DIR=pool_dir)
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import synth
        env = bench.dist_env()
        mx = bench.max_over_ranks(1.5 * (rank + 1), world)
        rate = bench.whole_job_rate(100.0, 0.5 + rank, world)  # the slowest rank took 1.5 s
        bench.barrier(world)
        sh = synth.Shape(L=2, E=4, k=2, H=64, F=64)
        mm, path = bench.shared_pool_file(sh, 3, world, rank)
        want = np.empty(sh.L * sh.E * sh.record_bytes, np.uint8)
        synth.fill_host_pool(want, sh, 3)
        same = bool(np.array_equal(np.asarray(mm), want))

        class Args:
            warmup, steps, cpu_seconds = 3, 2, 0.05

        idle = bench.run_reference(Args, rank, world) is None if rank > 0 else True
        out.put((rank, env, mx, rate, same, idle, path))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, str(tmp_path), out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, mx, rate, same, idle, path in res:
        assert env == (rank, 2, rank)
        assert mx == 3.0
        assert abs(rate - 2 * 100.0 / 1.5) < 1e-9
        assert same, "shared pool file differs from the seeded records"
        assert idle, "the reference arm did work on a rank other than 0"
        assert os.path.dirname(path) == str(tmp_path)
