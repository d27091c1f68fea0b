"""The benchmark's multi-process path (one process per GPU, weak scaling,
no data-path collective): timing is combined as the maximum over ranks
and every rank joins the barriers.  Run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    bench.barrier(w)
    elapsed = 10.0 + 5.0 * r  # rank 1 is the slowest
    q.put((r, bench.max_over_ranks(elapsed, w)))
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_single_process_env_defaults(monkeypatch):
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_step_accounting_counts_shared_blocks_once():
    import bench
    from workloads import draw_plan
    plan = draw_plan("smollm2-135m")
    acc = bench.step_accounting(plan)
    sh = plan.shape
    row = sh.n_kv * sh.head_dim * sh.itemsize
    logical = int(plan.seq_lens.sum()) * row * 2
    shared = 32 * row * 2 * (plan.num_seqs - 1)  # 2 shared blocks counted once
    assert acc["decode_kv_bytes"] == logical - shared
