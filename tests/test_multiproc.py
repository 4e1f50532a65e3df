"""The path partitions by request: two gloo ranks on CPU, each running the
oracle's swap-in and verify over its own half of the requests, reproduce the
single-process result, and bench.py's step-time reduction takes the maximum
over ranks. No collective is needed on the data path (only the barrier and
the timing reduction bench.py uses)."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads as W
from oracle import hs_oracle as O


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _run_requests(reqs, cfg, hb_np, pool, topk, clen, logits, drafts, skv):
    """Swap-in + verify for the given request ids with a private buffer."""
    idx = {b: i for i, b in enumerate(reqs)}
    rows = [r for r in range(cfg.R) if r // (cfg.d + 1) in idx]
    local_req = np.array([idx[r // (cfg.d + 1)] for r in rows])
    buf = O.HotBuffer(len(reqs), cfg.S, cfg.d + 1, hb_np["max_ctx"], cfg.block_size,
                      hb_np["hbt"][reqs], pool.clone())
    L = [cfg.L[b] for b in reqs]
    # one row per request (wave 0) keeps within the slot budget
    wave = [k for k, r in enumerate(rows) if r % (cfg.d + 1) == 0]
    out, valid, st, _ = buf.swap_in(local_req[wave], clen[np.array(rows)[wave]], L,
                                    topk[np.array(rows)[wave]])
    acc, nxt, Lnew, st2 = O.verify_finalize(buf, logits[reqs], drafts[reqs], skv[reqs], L)
    return {"out": out, "acc": acc, "nxt": nxt, "L": Lnew, "status": st | st2}


def _setup():
    cfg = W.get_config(1)
    cfg.B = 4
    cfg.L = [512, 300, 400, 64]
    req, ri = W.rows_of(cfg)
    hb = W.host_backed_case(cfg, device="cpu", extra_positions=8)
    topk = W.topk_independent(cfg, 0, cfg.L, req, ri)
    clen = W.causal_lengths(cfg.L, req, ri)
    logits, drafts, _ = W.planted_logits(cfg)
    skv = W.step_kv(cfg, 0, device="cpu")
    return cfg, {"max_ctx": hb["max_ctx"], "hbt": hb["hbt_np"]}, hb["pool"], topk, clen, \
        logits, drafts, skv


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg, hb, pool, topk, clen, logits, drafts, skv = _setup()
    mine = [b for b in range(cfg.B) if b % world == rank]
    res = _run_requests(mine, cfg, hb, pool, topk, clen, logits, drafts, skv)
    gathered = [None] * world
    dist.all_gather_object(gathered, (mine, res))
    t = torch.tensor([1.0 + rank])
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    if rank == 0:
        q.put((gathered, float(t.item())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_reproduce_single_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered, tmax = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert tmax == 2.0
    cfg, hb, pool, topk, clen, logits, drafts, skv = _setup()
    for mine, res in gathered:
        ref = _run_requests(mine, cfg, hb, pool, topk, clen, logits, drafts, skv)
        for k in ("out", "acc", "nxt", "L"):
            assert np.array_equal(res[k], ref[k])
    # and the per-request results equal those of one process holding all requests
    full = _run_requests(list(range(cfg.B)), cfg, hb, pool, topk, clen, logits, drafts, skv)
    for mine, res in gathered:
        for i, b in enumerate(mine):
            assert res["acc"][i] == full["acc"][b] and res["nxt"][i] == full["nxt"][b]
            assert res["L"][i] == full["L"][b]
