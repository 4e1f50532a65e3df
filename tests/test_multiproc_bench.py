"""bench.py's launch path for N > 1, on two gloo ranks on CPU: the rank
environment, the per-rank batch seed (each rank its own batch of the same
shape, weak scaling), the barrier, the max-over-ranks step time and the
whole-job throughput ws * rows / t. The data path has no collective."""
import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp

import bench
import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    ws, r, local = bench._dist()
    bench.init_dist(ws)
    cfg = W.get_config(2)
    cfg.seed = bench.rank_seed(cfg.seed, r)
    req, ri = W.rows_of(cfg)
    topk = W.topk_independent(cfg, 0, cfg.L, req, ri)[:4]     # the first request's rows
    bench.barrier(ws)
    t_local = [0.25, 0.375][r]                                 # this rank's step time, ms
    t_job = bench.max_over_ranks(t_local, ws)
    rows = bench.job_rows_per_s(ws, cfg.R, t_job)
    q.put((r, ws, local, cfg.seed, topk, t_job, rows))
    bench.barrier(ws)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_bench_rank_logic_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(k, 2, port, q)) for k in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ws0, l0, s0, tk0, t0, v0), (r1, ws1, l1, s1, tk1, t1, v1) = res
    assert (r0, r1) == (0, 1) and ws0 == ws1 == 2 and (l0, l1) == (0, 1)
    base = W.get_config(2).seed
    assert s0 == base and s1 == base + 1000
    assert tk0.shape == tk1.shape and not np.array_equal(tk0, tk1)   # own batch, same shape
    assert t0 == t1 == 0.375                                         # the slower rank's time
    assert v0 == v1 == 2 * 128 / 0.375e-3


def test_single_rank_helpers():
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.job_rows_per_s(1, 128, 0.1) == 128 / 1e-4
    assert bench.rank_seed(2, 0) == 2 and bench.rank_seed(2, 3) == 3002
