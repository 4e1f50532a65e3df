"""GPU parity of hs_swap_in_attn_decode: the swap-in and the attention of a
step in one call, the copies of later row groups overlapped with the
attention of earlier ones. It must give bit for bit what hs_swap_in followed
by hs_sparse_attn_decode gives on a twin buffer (slot tables, valid counts,
statistics, status, maps, timestamps, hot rows, out and lse), and its
attention must match the oracle's on sampled rows."""
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


def _same_state(hs, b1, b2, hot1, hot2, S_tot, S, reqs):
    d1, d2 = b1.dump(), b2.dump()
    for x, y in zip(d1, d2):
        assert torch.equal(x, y)
    h1 = hot1.view(torch.int16).view(-1, S_tot, 576)[:, :S]
    h2 = hot2.view(torch.int16).view(-1, S_tot, 576)[:, :S]
    assert torch.equal(h1[reqs], h2[reqs])
    assert b1.clock == b2.clock


def test_workload4_fused_step_matches_serial_and_oracle():
    """Workload 4 (128 requests, contexts 16K-128K, 512 rows, 90 % reuse), 4
    decode steps on two buffers: serial calls on one, the fused call with the
    library's row groups on the other. Every output agrees bit for bit every
    step; requests 3, 19, ..., 115 are followed by the oracle, whose attention
    over its own hot buffer must match the fused call's on their rows."""
    hs = lib()
    cfg = W.get_config(4)
    steps = 4
    req, ri = W.rows_of(cfg)
    clen = W.causal_lengths(cfg.L, req, ri)
    hb = W.host_backed_case(cfg, device=DEV)
    hot2 = torch.zeros_like(hb["hot"])
    mk = lambda hot: hs.HsBuffer(cfg.B, cfg.S, cfg.d + 1, hb["max_ctx"], cfg.block_size, hot,
                                 hb["pool"], hb["hbt"])
    b_ser, b_fus = mk(hb["hot"]), mk(hot2)
    groups = hs.hs_step_groups(cfg.R, cfg.H)
    assert len(groups) >= 2 and groups[-1] == cfg.R
    sample = list(range(3, cfg.B, 16))
    ref = O.HotBuffer(cfg.B, cfg.S, cfg.d + 1, hb["max_ctx"], cfg.block_size, hb["hbt_np"],
                      hb["pool"])
    rows_s = np.where(np.isin(req, sample))[0]
    sets = [W.locality_sets(cfg, cfg.L[b], b, steps) for b in range(cfg.B)]
    t_req, t_clen = _t(req), _t(clen)
    st1 = torch.zeros(2, dtype=torch.int64, device=DEV)
    st2 = torch.zeros_like(st1)
    for step in range(steps):
        topk_np = W.topk_shared_sets(cfg, sets, step)
        topk = _t(topk_np)
        q = W.step_q(cfg, step, device=DEV)
        outs = []
        for which in ("serial", "fused"):
            idx = torch.full((cfg.R, cfg.K), 7, dtype=torch.int32, device=DEV)
            valid = torch.full((cfg.R,), 7, dtype=torch.int32, device=DEV)
            out = torch.empty((cfg.R, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
            lse = torch.empty((cfg.R, cfg.H), dtype=torch.float32, device=DEV)
            if which == "serial":
                hs.hs_swap_in(b_ser, t_req, t_clen, hb["kv_len"], topk, idx, valid, st1)
                hs.hs_sparse_attn_decode(q, hb["hot"], idx, cfg.scale, out, lse)
            else:
                hs.hs_swap_in_attn_decode(b_fus, t_req, t_clen, hb["kv_len"], topk, q,
                                          cfg.scale, idx, out, out_valid=valid, lse=lse,
                                          stats=st2)
            torch.cuda.synchronize()
            outs.append((idx, valid, out, lse))
        (i1, v1, o1, l1), (i2, v2, o2, l2) = outs
        assert torch.equal(i1, i2) and torch.equal(v1, v2)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
        assert torch.equal(st1, st2)
        assert hs.hs_get_status(b_ser) == hs.hs_get_status(b_fus) == 0
        # the oracle on the sampled requests' rows of the same call
        e_out, e_valid, e_st, _ = ref.swap_in(req[rows_s], clen[rows_s], cfg.L, topk_np[rows_s])
        assert ref.now == b_fus.clock
        assert np.array_equal(np_(i2)[rows_s], e_out)
        assert np.array_equal(np_(v2)[rows_s], e_valid)
        qc = q[torch.as_tensor(rows_s, device=DEV)].cpu()
        r_out, r_lse = O.sparse_attn_decode_rows(
            qc, lambda sel: O.bf16_bits_to_f64(ref.hot[np.asarray(sel)]), e_out, cfg.scale,
            range(len(rows_s)))
        check_attn(o2, np.stack([r_out[k] for k in range(len(rows_s))]), l2,
                   np.stack([r_lse[k] for k in range(len(rows_s))]), rows=rows_s)
    assert st2[1].item() > 0
    _same_state(hs, b_ser, b_fus, hb["hot"], hot2, cfg.S + cfg.d + 1, cfg.S,
                torch.arange(cfg.B, device=DEV))


@pytest.mark.parametrize("seed,H", [(0, 32), (1, 32), (2, 32), (3, 32), (4, 200)])
def test_explicit_groups_scattered_rows(seed, H):
    """Rows of a request scattered over the call and over several groups (a
    request is swapped in with the group of its first row), random group
    ends, 1 to 8 groups, evictions and step positions: bit for bit the serial
    calls on a twin buffer, and the attention matches the oracle on every
    row. H = 200: two head groups per row, the last ragged."""
    hs = lib()
    g = np.random.default_rng(500 + seed)
    B, S, n_step, bs, max_ctx = 6, 40, 3, 4, 160
    nblk = max_ctx // bs
    hbt = g.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    pool = W.host_pool_tensor(B * nblk * bs, 900 + seed, device=DEV)
    hots = [torch.zeros((B * (S + n_step), 576), dtype=torch.bfloat16, device=DEV)
            for _ in range(2)]
    bufs = [hs.HsBuffer(B, S, n_step, max_ctx, bs, h, pool, _t(hbt)) for h in hots]
    ref = O.HotBuffer(B, S, n_step, max_ctx, bs, hbt, pool.clone())
    # a follower layer of each buffer, filled by repeating each call's plan
    f_pool = W.host_pool_tensor(B * nblk * bs, 950 + seed, device=DEV)
    f_hots = [torch.zeros_like(hots[0]) for _ in range(2)]
    L = [int(x) for x in g.integers(60, 150, size=B)]
    kv_len = _t(np.asarray(L, np.int32))
    for call in range(6):
        R = int(g.integers(1, 40))
        req = g.integers(0, B, size=R).astype(np.int32)
        K = int(g.integers(1, 48))
        clen = np.array([L[b] + int(g.integers(1, n_step + 1)) for b in req], np.int32)
        topk = np.stack([g.integers(-1, c + 1, size=K) for c in clen]).astype(np.int32)
        n_groups = int(g.integers(1, min(8, R) + 1))
        ends = sorted(g.choice(np.arange(1, R), n_groups - 1, replace=False).tolist()) + [R] \
            if n_groups > 1 else [R]
        q = (torch.randn((R, H, 576), generator=torch.Generator().manual_seed(call + 10 * seed))
             * 0.5).to(torch.bfloat16).to(DEV)
        res = []
        for k, buf in enumerate(bufs):
            idx = torch.full((R, K), 7, dtype=torch.int32, device=DEV)
            valid = torch.full((R,), 7, dtype=torch.int32, device=DEV)
            out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=DEV)
            lse = torch.empty((R, H), dtype=torch.float32, device=DEV)
            if k == 0:
                hs.hs_swap_in(buf, _t(req), _t(clen), kv_len, _t(topk), idx, valid)
                hs.hs_sparse_attn_decode(q, hots[0], idx, 0.07, out, lse)
            else:
                hs.hs_swap_in_attn_decode(buf, _t(req), _t(clen), kv_len, _t(topk), q, 0.07, idx,
                                          out, groups=ends, out_valid=valid, lse=lse)
            hs.hs_swap_apply_plan(buf, [f_hots[k]], [f_pool])
            torch.cuda.synchronize()
            res.append((idx, valid, out, lse))
        (i1, v1, o1, l1), (i2, v2, o2, l2) = res
        assert torch.equal(i1, i2) and torch.equal(v1, v2)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
        e_out, e_valid, e_st, _ = ref.swap_in(req, clen, L, topk)
        assert np.array_equal(np_(i2), e_out) and np.array_equal(np_(v2), e_valid)
        assert hs.hs_get_status(bufs[1]) == hs.hs_get_status(bufs[0]) == e_st
        r_out, r_lse = O.sparse_attn_decode_rows(
            q.cpu(), lambda sel: O.bf16_bits_to_f64(ref.hot[np.asarray(sel)]), e_out, 0.07,
            range(R))
        check_attn(o2, np.stack([r_out[k] for k in range(R)]), l2,
                   np.stack([r_lse[k] for k in range(R)]))
    _same_state(hs, bufs[0], bufs[1], hots[0], hots[1], S + n_step, S,
                torch.arange(B, device=DEV))
    assert torch.equal(f_hots[0].view(torch.int16), f_hots[1].view(torch.int16))


def test_fused_step_in_a_cuda_graph():
    """The call captured in a CUDA graph (its own streams fork from and join
    the capturing stream) gives, replay after replay over new top-k and q,
    what the serial calls captured in another graph give on a twin buffer.
    (A replay stamps the LRU clock of its capture, so both sides are graphs.)"""
    hs = lib()
    g = np.random.default_rng(77)
    B, S, n_step, bs, max_ctx, H, K = 8, 128, 2, 8, 512, 64, 48
    nblk = max_ctx // bs
    hbt = g.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    pool = W.host_pool_tensor(B * nblk * bs, 78, device=DEV)
    hots = [torch.zeros((B * (S + n_step), 576), dtype=torch.bfloat16, device=DEV)
            for _ in range(2)]
    bufs = [hs.HsBuffer(B, S, n_step, max_ctx, bs, h, pool, _t(hbt)) for h in hots]
    L = [400] * B
    req = np.repeat(np.arange(B, dtype=np.int32), n_step)
    clen = np.array([L[b] + 1 + (i % n_step) for i, b in enumerate(req)], np.int32)
    R = len(req)
    t_req, t_clen, kv_len = _t(req), _t(clen), _t(np.asarray(L, np.int32))
    topk = torch.empty((R, K), dtype=torch.int32, device=DEV)
    q = torch.empty((R, H, 576), dtype=torch.bfloat16, device=DEV)
    idx = [torch.empty((R, K), dtype=torch.int32, device=DEV) for _ in range(2)]
    out = [torch.empty((R, H, 512), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    ends = [4, 10, R]

    def new_inputs():
        topk.copy_(_t(np.stack([g.choice(c, K, replace=False) for c in clen]).astype(np.int32)))
        q.normal_()

    def serial(st):
        hs.hs_swap_in(bufs[0], t_req, t_clen, kv_len, topk, idx[0], stream=st)
        hs.hs_sparse_attn_decode(q, hots[0], idx[0], 0.05, out[0], stream=st)

    def fused(st):
        hs.hs_swap_in_attn_decode(bufs[1], t_req, t_clen, kv_len, topk, q, 0.05, idx[1], out[1],
                                  groups=ends, stream=st)

    # one eager call of each first (first-call attributes are set outside capture)
    new_inputs()
    serial(None)
    fused(None)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graphs = [torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()]
    with torch.cuda.stream(s):
        for gr, fn in zip(graphs, (serial, fused)):
            with torch.cuda.graph(gr, stream=s):
                fn(s)
    for step in range(4):
        new_inputs()
        graphs[0].replay()
        graphs[1].replay()
        torch.cuda.synchronize()
        assert torch.equal(idx[0], idx[1])
        assert torch.equal(out[0].view(torch.int16), out[1].view(torch.int16))
    assert hs.hs_get_status(bufs[1]) == hs.hs_get_status(bufs[0]) == 0
    _same_state(hs, bufs[0], bufs[1], hots[0], hots[1], S + n_step, S,
                torch.arange(B, device=DEV))


def test_bad_groups_are_refused_before_any_work():
    hs = lib()
    B, S, n_step, bs, max_ctx = 2, 8, 2, 4, 32
    hbt = np.arange(B * 8, dtype=np.int32).reshape(B, 8)
    pool = W.host_pool_tensor(B * 32, 5, device=DEV)
    hot = torch.zeros((B * (S + n_step), 576), dtype=torch.bfloat16, device=DEV)
    buf = hs.HsBuffer(B, S, n_step, max_ctx, bs, hot, pool, _t(hbt))
    R, K, H = 4, 3, 16
    req = _t(np.array([0, 0, 1, 1], np.int32))
    clen = _t(np.array([21, 22, 21, 22], np.int32))
    kv_len = _t(np.array([20, 20], np.int32))
    topk = _t(np.array([[1, 2, 3]] * 4, np.int32))
    q = torch.zeros((R, H, 576), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((R, K), dtype=torch.int32, device=DEV)
    out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=DEV)
    c0 = buf.clock
    for bad in ([2, 2, 4], [0, 4], [3], [1, 2, 3, 4, 4], list(range(1, 10))):
        with pytest.raises(hs.HisparseError):
            hs.hs_swap_in_attn_decode(buf, req, clen, kv_len, topk, q, 0.1, idx, out, groups=bad)
    assert buf.clock == c0
    hs.hs_swap_in_attn_decode(buf, req, clen, kv_len, topk, q, 0.1, idx, out, groups=[1, 3, 4])
    torch.cuda.synchronize()
    assert buf.clock == c0 + 1 and hs.hs_get_status(buf) == 0


@pytest.mark.parametrize("max_reqs,copy_sms", [(1000, 0), (12, 3)])
def test_large_buffer_and_held_copy_kernels(max_reqs, copy_sms):
    """A buffer of 1000 requests (the copy kernel's per-request prefix no
    longer fits beside an attention block, so later groups' copies wait for
    free SMs) and a buffer whose copy kernels are held to 3 SMs: three calls
    of scattered rows in four groups, bit for bit the serial pair."""
    hs = lib()
    g = np.random.default_rng(800 + max_reqs)
    S, n_step, bs, max_ctx, H, K = 16, 2, 8, 128, 32, 12
    nblk = max_ctx // bs
    hbt = g.permutation(max_reqs * nblk).reshape(max_reqs, nblk).astype(np.int32)
    pool = W.host_pool_tensor(max_reqs * nblk * bs, 801, device=DEV)
    hots = [torch.zeros((max_reqs * (S + n_step), 576), dtype=torch.bfloat16, device=DEV)
            for _ in range(2)]
    bufs = [hs.HsBuffer(max_reqs, S, n_step, max_ctx, bs, h, pool, _t(hbt)) for h in hots]
    for buf in bufs:
        hs.hs_buffer_set_copy_sms(buf, copy_sms)
    L = [int(x) for x in g.integers(20, 100, size=max_reqs)]
    kv_len = _t(np.asarray(L, np.int32))
    for call in range(3):
        R = 40
        req = g.choice(max_reqs, R).astype(np.int32)
        clen = np.array([L[b] + int(g.integers(1, n_step + 1)) for b in req], np.int32)
        topk = np.stack([g.choice(c, K, replace=False) for c in clen]).astype(np.int32)
        q = (torch.randn((R, H, 576), generator=torch.Generator().manual_seed(call))
             * 0.5).to(torch.bfloat16).to(DEV)
        res = []
        for k, buf in enumerate(bufs):
            idx = torch.empty((R, K), dtype=torch.int32, device=DEV)
            out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=DEV)
            if k == 0:
                hs.hs_swap_in(buf, _t(req), _t(clen), kv_len, _t(topk), idx)
                hs.hs_sparse_attn_decode(q, hots[0], idx, 0.05, out)
            else:
                hs.hs_swap_in_attn_decode(buf, _t(req), _t(clen), kv_len, _t(topk), q, 0.05, idx,
                                          out, groups=[5, 17, 30, R])
            torch.cuda.synchronize()
            res.append((idx, out))
        assert torch.equal(res[0][0], res[1][0])
        assert torch.equal(res[0][1].view(torch.int16), res[1][1].view(torch.int16))
        # requests drawn more than once may overflow their slots: the same
        # capacity bits on both sides
        assert hs.hs_get_status(bufs[0]) == hs.hs_get_status(bufs[1])
    _same_state(hs, bufs[0], bufs[1], hots[0], hots[1], S + n_step, S,
                torch.arange(max_reqs, device=DEV))


def test_degenerate_calls_match_the_serial_pair():
    """K = 0 (every row without keys: out 0, lse -inf) and R = 0 (nothing but
    the clock) give what the serial pair gives on a twin buffer."""
    hs = lib()
    B, S, n_step, bs, max_ctx, H = 3, 8, 2, 4, 32, 16
    hbt = np.arange(B * 8, dtype=np.int32).reshape(B, 8)
    pool = W.host_pool_tensor(B * 32, 6, device=DEV)
    hots = [torch.zeros((B * (S + n_step), 576), dtype=torch.bfloat16, device=DEV)
            for _ in range(2)]
    bufs = [hs.HsBuffer(B, S, n_step, max_ctx, bs, h, pool, _t(hbt)) for h in hots]
    kv_len = _t(np.array([20, 20, 20], np.int32))
    for R, K in ((5, 0), (0, 4)):
        req = _t(np.arange(R, dtype=np.int32) % B)
        clen = _t(np.full(R, 21, np.int32))
        topk = torch.zeros((R, K), dtype=torch.int32, device=DEV)
        q = torch.ones((R, H, 576), dtype=torch.bfloat16, device=DEV)
        res = []
        for k, buf in enumerate(bufs):
            idx = torch.full((R, K), 7, dtype=torch.int32, device=DEV)
            out = torch.full((R, H, 512), 3.0, dtype=torch.bfloat16, device=DEV)
            lse = torch.zeros((R, H), dtype=torch.float32, device=DEV)
            if k == 0:
                hs.hs_swap_in(buf, req, clen, kv_len, topk, idx)
                hs.hs_sparse_attn_decode(q, hots[0], idx, 0.1, out, lse)
            else:
                hs.hs_swap_in_attn_decode(buf, req, clen, kv_len, topk, q, 0.1, idx, out, lse=lse)
            torch.cuda.synchronize()
            res.append((out, lse))
        assert torch.equal(res[0][0].view(torch.int16), res[1][0].view(torch.int16))
        assert torch.equal(res[0][1].view(torch.int32), res[1][1].view(torch.int32))
        if R:
            assert (res[1][0].float() == 0).all() and torch.isneginf(res[1][1]).all()
        assert bufs[0].clock == bufs[1].clock
        assert hs.hs_get_status(bufs[0]) == hs.hs_get_status(bufs[1]) == 0


def test_library_groups():
    """The split: the first group one attention wave, the other rows in at
    most 7 groups of equal size, a whole number of waves, the last taking
    what is left; ends rising to R."""
    hs = lib()
    wave = hs.hs_step_groups(100000, 128)[0]
    assert wave >= 1
    assert hs.hs_step_groups(100000, 256)[0] == max(1, wave // 2)
    for R, H in ((1, 128), (wave, 128), (wave + 1, 128), (512, 128), (100000, 128),
                 (512, 256), (40, 16)):
        ends = hs.hs_step_groups(R, H)
        w = hs.hs_step_groups(100000, H)[0]
        assert 1 <= len(ends) <= 8 and ends[-1] == R
        assert all(a < b for a, b in zip(ends, ends[1:]))
        sizes = np.diff([0] + ends)
        assert sizes[0] == min(R, w)
        if len(sizes) > 2:
            mid = sizes[1:-1]
            assert (mid == mid[0]).all() and mid[0] % w == 0 and 0 < sizes[-1] <= mid[0]
    assert hs.hs_step_groups(0, 128) == []


def test_copy_block_fits_beside_attention():
    """The later groups' copies overlap the attention only when a copy block
    fits on an SM beside an attention CTA (register-file quarters, shared
    memory, threads). A kernel change that breaks this still passes every
    bit-exactness test, so it is checked here: it holds for buffers of up to
    448 requests and fails for 16384 (a 64 KB copy-prefix table)."""
    hs = lib()
    for max_reqs in (1, 64, 128, 448):
        assert hs.hs_step_overlap_fits(max_reqs), max_reqs
    assert not hs.hs_step_overlap_fits(16384)
