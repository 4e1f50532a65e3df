"""GPU parity of a2-a5 (swap-in): slot tables, valid counts, status bits, the
position <-> slot maps, timestamps and hot-buffer rows match the oracle
bit-exactly after every call."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import hs_oracle as O
from gpu_util import check_attn, lib, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a):
    return torch.as_tensor(np.ascontiguousarray(a), device=DEV)


class Pair:
    """The GPU buffer and the oracle buffer over the same inputs (copy_sms >
    0: the swap-in's copy kernel held to about that many SMs)."""

    def __init__(self, B, S, n_step, max_ctx, bs, seed, copy_sms=0):
        hs = lib()
        g = np.random.default_rng(seed)
        nblk = (max_ctx + bs - 1) // bs
        self.hbt = g.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
        self.pool = W.host_pool_tensor(B * nblk * bs, seed, device=DEV)
        self.hot = torch.zeros((B * (S + n_step), 576), dtype=torch.bfloat16, device=DEV)
        self.buf = hs.HsBuffer(B, S, n_step, max_ctx, bs, self.hot, self.pool, _t(self.hbt))
        if copy_sms:
            hs.hs_buffer_set_copy_sms(self.buf, copy_sms)
        self.ref = O.HotBuffer(B, S, n_step, max_ctx, bs, self.hbt, self.pool.clone())
        self.B, self.S, self.n_step = B, S, n_step
        self.hs = hs
        self.stats = torch.zeros(2, dtype=torch.int64, device=DEV)

    def call(self, req, clen, L, topk):
        R, K = topk.shape
        out = torch.full((R, K), 9, dtype=torch.int32, device=DEV)
        valid = torch.full((R,), 9, dtype=torch.int32, device=DEV)
        kv_len = _t(np.asarray(L, np.int32))
        self.hs.hs_swap_in(self.buf, _t(req), _t(clen), kv_len, _t(topk), out, valid,
                           self.stats)
        e_out, e_valid, e_st, e_stats = self.ref.swap_in(req, clen, L, topk)
        st = self.hs.hs_get_status(self.buf)
        assert np.array_equal(np_(out), e_out)
        assert np.array_equal(np_(valid), e_valid)
        assert st == e_st
        return e_stats

    def compare_state(self, reqs=None):
        ts, stok, sts = self.buf.dump()
        reqs = range(self.B) if reqs is None else reqs
        hot = self.hot.view(torch.int16).cpu().numpy().view(np.uint16)
        for b in reqs:
            assert stok[b].tolist() == self.ref.slot_token[b]
            assert sts[b].tolist() == self.ref.slot_ts[b]
            assert np.array_equal(ts[b].numpy(), self.ref.token_slot_array(b))
            lo = b * self.ref.S_tot
            assert np.array_equal(hot[lo:lo + self.S], self.ref.hot[lo:lo + self.S])
        assert self.buf.clock == self.ref.now


@pytest.mark.parametrize("copy_sms", [0, 3])
@pytest.mark.parametrize("seed", range(6))
def test_random_sequences_tiny(seed, copy_sms):
    g = np.random.default_rng(1000 + seed)
    B, S, n_step, bs, max_ctx = 3, int(g.integers(2, 12)), 3, 4, 48
    p = Pair(B, S, n_step, max_ctx, bs, seed, copy_sms)
    L = [int(x) for x in g.integers(1, 44, size=B)]
    for call in range(12):
        R = int(g.integers(1, 6))
        req = g.integers(0, B, size=R).astype(np.int32)
        K = int(g.integers(1, 40))
        clen = np.array([L[b] + int(g.integers(1, n_step + 1)) for b in req], np.int32)
        topk = np.stack([g.integers(-2, c + 2, size=K) for c in clen]).astype(np.int32)
        p.call(req, clen, L, topk)
        p.compare_state()


def test_capacity_overflow_leaves_request_unchanged():
    p = Pair(2, 4, 1, 64, 8, 7)
    L = [60, 60]
    p.call(np.array([0, 1], np.int32), np.array([61, 61], np.int32), L,
           np.array([[1, 2, 3, -1, -1], [5, 6, -1, -1, -1]], np.int32))
    # request 0 now needs 5 distinct positions > S = 4
    p.call(np.array([0, 0, 1], np.int32), np.array([61, 61, 61], np.int32), L,
           np.array([[1, 9, 10, 60, -1], [11, 12, 2, -1, -1], [6, 7, -1, -1, -1]], np.int32))
    p.compare_state()


def test_many_rows_one_request_dedup_and_large_K():
    g = np.random.default_rng(9)
    p = Pair(2, 1024, 4, 4096, 64, 9)
    L = [4000, 3000]
    req = np.array([0, 0, 0, 0, 1, 1, 1, 1], np.int32)
    clen = np.array([L[b] + 1 + i % 4 for i, b in enumerate(req)], np.int32)
    base = [g.choice(L[0], 700, replace=False), g.choice(L[1], 900, replace=False)]
    for step in range(3):
        topk = np.stack([g.permutation(base[b])[:600] for b in req]).astype(np.int32)
        p.call(req, clen, L, topk)
        p.compare_state()
        base = [np.concatenate([x[:500], g.choice(L[i], 200, replace=False)])
                for i, x in enumerate(base)]


def test_resolve_and_swap_paths_give_identical_attention():
    """The two residency paths ("vllm 分析(十二) HiSparse 下篇", resolve_topk: fully
    resident index conversion versus swap-in) must feed attention the same
    rows in the same order, so the outputs are bit-identical."""
    hs = lib()
    cfg = W.get_config(1)
    req, ri = W.rows_of(cfg)
    hb = W.host_backed_case(cfg, device=DEV, extra_positions=8)
    buf = hs.HsBuffer(cfg.B, cfg.S, cfg.d + 1, hb["max_ctx"], cfg.block_size, hb["hot"],
                      hb["pool"], hb["hbt"])
    pool_dev = hb["pool"].to(DEV)
    # step slots hold the same rows as the paged pool for positions L .. L+d
    for b in range(cfg.B):
        for i in range(cfg.d + 1):
            t = cfg.L[b] + i
            row = int(hb["hbt_np"][b, t // cfg.block_size]) * cfg.block_size + t % cfg.block_size
            hb["hot"][b * hb["S_tot"] + cfg.S + i] = pool_dev[row]
    topk = W.topk_independent(cfg, 0, cfg.L, req, ri)
    clen = W.causal_lengths(cfg.L, req, ri)
    q = W.step_q(cfg, 0, device=DEV)
    for wave in range(cfg.d + 1):
        rows = np.where(ri == wave)[0]
        tk, rq, cl = _t(topk[rows]), _t(req[rows]), _t(clen[rows])
        a = torch.empty_like(tk)
        hs.hs_swap_in(buf, rq, cl, hb["kv_len"], tk, a)
        b_ = torch.empty_like(tk)
        hs.hs_resolve_topk(rq, cl, hb["hbt"], tk, cfg.block_size, cfg.block_size, b_)
        qq = q[_t(rows)].contiguous()
        o1 = torch.empty((len(rows), cfg.H, 512), dtype=torch.bfloat16, device=DEV)
        o2 = torch.empty_like(o1)
        hs.hs_sparse_attn_decode(qq, hb["hot"], a, cfg.scale, o1)
        hs.hs_sparse_attn_decode(qq, pool_dev, b_, cfg.scale, o2)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
    assert hs.hs_get_status(buf) == 0


def _run_locality(cfg_no, sample, steps=None, copy_sms=0, attn=True):
    """Workload 3 or 4 over its decode steps: every swap-in call on all the
    workload's rows; the oracle follows the sampled requests (their rows of
    the same calls). After every call the sampled rows' slot tables and valid
    counts must match bit for bit, and (attn) the attention over the GPU's
    hot buffer with the GPU's slot tables must match the oracle's attention
    over its own hot buffer with its own tables (R13); at the end the sampled
    requests' maps, timestamps and hot rows must match bit for bit."""
    hs = lib()
    cfg = W.get_config(cfg_no)
    steps = steps or cfg.steps
    req, ri = W.rows_of(cfg)
    clen = W.causal_lengths(cfg.L, req, ri)
    hb = W.host_backed_case(cfg, device=DEV)
    buf = hs.HsBuffer(cfg.B, cfg.S, cfg.d + 1, hb["max_ctx"], cfg.block_size, hb["hot"],
                      hb["pool"], hb["hbt"])
    if copy_sms:
        hs.hs_buffer_set_copy_sms(buf, copy_sms)
    ref = O.HotBuffer(cfg.B, cfg.S, cfg.d + 1, hb["max_ctx"], cfg.block_size, hb["hbt_np"],
                      hb["pool"])
    sets = [W.locality_sets(cfg, cfg.L[b], b, steps) for b in range(cfg.B)]
    rows_s = np.where(np.isin(req, sample))[0]
    t_rows = torch.as_tensor(rows_s, device=DEV)
    stats = torch.zeros(2, dtype=torch.int64, device=DEV)
    for step in range(steps):
        topk = W.topk_shared_sets(cfg, sets, step)
        out = torch.empty((cfg.R, cfg.K), dtype=torch.int32, device=DEV)
        valid = torch.empty((cfg.R,), dtype=torch.int32, device=DEV)
        hs.hs_swap_in(buf, _t(req), _t(clen), hb["kv_len"], _t(topk), out, valid, stats)
        e_out, e_valid, e_st, _ = ref.swap_in(req[rows_s], clen[rows_s], cfg.L, topk[rows_s])
        assert ref.now == buf.clock   # the oracle saw the sampled rows of the same calls
        assert np.array_equal(np_(out)[rows_s], e_out)
        assert np.array_equal(np_(valid)[rows_s], e_valid)
        assert hs.hs_get_status(buf) == e_st == 0
        if attn:
            q = W.step_q(cfg, step, device=DEV)[t_rows].contiguous()
            o = torch.empty((len(rows_s), cfg.H, 512), dtype=torch.bfloat16, device=DEV)
            lse = torch.empty((len(rows_s), cfg.H), dtype=torch.float32, device=DEV)
            hs.hs_sparse_attn_decode(q, hb["hot"], out[t_rows].contiguous(), cfg.scale, o, lse)
            qc = q.cpu()
            outs, lses = O.sparse_attn_decode_rows(
                qc, lambda sel: O.bf16_bits_to_f64(ref.hot[np.asarray(sel)]), e_out, cfg.scale,
                range(len(rows_s)))
            check_attn(o, np.stack([outs[k] for k in range(len(rows_s))]), lse,
                       np.stack([lses[k] for k in range(len(rows_s))]))
    ts, stok, sts = buf.dump()
    hot = hb["hot"].view(torch.int16).cpu().numpy().view(np.uint16)
    for b in sample:
        assert stok[b].tolist() == ref.slot_token[b]
        assert sts[b].tolist() == ref.slot_ts[b]
        assert np.array_equal(ts[b].numpy(), ref.token_slot_array(b))
        lo = b * ref.S_tot
        assert np.array_equal(hot[lo:lo + cfg.S], ref.hot[lo:lo + cfg.S])
    return np_(stats)


def test_workload3_all_steps_every_eighth_request():
    """All 16 steps of workload 3; requests 0, 8, ..., 56 followed by the
    oracle, with the attention on their swap-in indices every step."""
    stats = _run_locality(3, sample=list(range(0, 64, 8)))
    assert stats[1] > 0


def test_workload3_sampled_requests_separate_copy_kernel():
    stats = _run_locality(3, sample=[1, 40], steps=3, copy_sms=16, attn=False)
    assert stats[1] > 0


def test_workload4_all_steps_every_eighth_request():
    """All 8 steps of workload 4 (contexts 16K-128K); requests 0, 8, ..., 120
    followed by the oracle, with the attention on their swap-in indices
    every step."""
    _run_locality(4, sample=list(range(0, 128, 8)))


def test_largest_slot_count_and_long_context():
    """S = 8192 (the largest slot count) and a 300,000-position context, past
    the bitmap limit of 262,144 positions, so claims go through epoch marks
    and the misses through the bitonic sort. Five calls of 3000 positions
    shared by both rows, half of them reused, fill the buffer and evict;
    every piece of state matches the oracle after each call."""
    g = np.random.default_rng(21)
    S, max_ctx, L = 8192, 300_000, 290_000
    p = Pair(1, S, 2, max_ctx, 64, 21)
    req = np.zeros(2, np.int32)
    clen = np.array([L + 1, L + 2], np.int32)
    cur = g.choice(L, 3000, replace=False)
    for call in range(5):
        topk = np.stack([g.permutation(cur), g.permutation(cur)]).astype(np.int32)
        p.call(req, clen, [L], topk)
        p.compare_state()
        fresh = np.setdiff1d(g.choice(L, 3000, replace=False), cur)[:1500]
        cur = np.concatenate([g.permutation(cur)[:3000 - len(fresh)], fresh])


def test_most_requests_per_buffer():
    """max_reqs = 16384, the limit (the gather's prefix over every request
    sits in shared memory, and the metadata launch has a block per request),
    with rows of three requests at the start, middle and end of the range."""
    g = np.random.default_rng(31)
    B, S, n_step, max_ctx, bs = 16384, 8, 2, 16, 4
    p = Pair(B, S, n_step, max_ctx, bs, 31)
    L = [10] * B
    active = [0, 8191, 16383]
    for call in range(3):
        req = np.array([0, 0, 8191, 16383, 16383], np.int32)
        clen = np.array([L[b] + 1 + (i % 2) for i, b in enumerate(req)], np.int32)
        topk = np.stack([g.choice(c, 6, replace=False) for c in clen]).astype(np.int32)
        p.call(req, clen, L, topk)
        p.compare_state(reqs=active)
