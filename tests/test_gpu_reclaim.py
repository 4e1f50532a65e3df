"""GPU parity of the switch from fully resident to host-backed ("vllm 分析(十二)
HiSparse 下篇", reclaim_resident_blocks and the fully_resident flag): the
reclaim kernel bit-exact against the oracle, the mixed-batch attention
against the oracle and bit-identical to the one-cache attention of each row,
and a request walked from the resident cache to swap-in while another stays
resident, its attention unchanged bit for bit."""
import numpy as np
import pytest
import torch

from oracle import hs_oracle as O
from gpu_util import check_attn, lib, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a):
    return torch.as_tensor(np.ascontiguousarray(a), device=DEV)


def _bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("B,stride", [(1, 1), (3, 6), (37, 9), (2500, 7)])
def test_reclaim_matches_oracle(B, stride):
    hs = lib()
    g = np.random.default_rng(B * 100 + stride)
    bt = g.permutation(B * stride).reshape(B, stride).astype(np.int32)
    bt[g.random((B, stride)) < 0.1] = -1
    nb = g.integers(-1, stride + 2, size=B).astype(np.int32)
    n_recl = len(O.reclaimable_pages(bt, nb))
    for need in sorted({0, 1, 5, n_recl // 2, n_recl, n_recl + 3}):
        d_bt = _t(bt)
        freed = torch.full((need,), 7, dtype=torch.int32, device=DEV)
        fully = torch.full((B,), 7, dtype=torch.int32, device=DEV)
        n = torch.full((1,), 7, dtype=torch.int32, device=DEV)
        hs.hs_reclaim_resident(d_bt, _t(nb), need, freed if need else None, fully, n)
        e_bt, e_freed, e_fully, e_n = O.reclaim_resident(bt, nb, need)
        torch.cuda.synchronize()
        assert np.array_equal(np_(d_bt), e_bt)
        assert np.array_equal(np_(freed), e_freed)
        assert np.array_equal(np_(fully), e_fully)
        assert int(n.item()) == e_n


def test_mixed_attention_matches_oracle_and_single_cache():
    hs = lib()
    g = np.random.default_rng(11)
    R, H, K, NA, NH = 7, 128, 300, 5000, 700
    q = _bf16(g.standard_normal((R, H, 576)) / 24).to(DEV)
    kv_a = _bf16(g.standard_normal((NA, 576)) / 24).to(DEV)
    kv_h = _bf16(g.standard_normal((NH, 576)) / 24).to(DEV)
    idx = g.integers(-1, NA, size=(R, K)).astype(np.int32)
    req = np.array([0, 1, 1, 2, 0, 2, 3], np.int32)
    fully = np.array([1, 0, 1, 0], np.int32)
    for r in range(R):                     # hot rows: mostly valid slots
        if fully[req[r]] == 0:
            idx[r, : K - 20] = g.integers(0, NH, size=K - 20)
    out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((R, H), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hs.hs_sparse_attn_decode_mixed(q, kv_a, kv_h, _t(req), _t(fully), _t(idx), 0.04, out, lse,
                                   st)
    ref, ref_lse = O.sparse_attn_decode_mixed(q.cpu(), kv_a.cpu(), kv_h.cpu(), req, fully, idx,
                                              0.04)
    torch.cuda.synchronize()
    check_attn(out, ref, lse, ref_lse)
    assert int(st.item()) == 0
    # each row comes out bit for bit as the one-cache call over its own cache
    for cache, sel in ((kv_a, fully[req] != 0), (kv_h, fully[req] == 0)):
        rows = np.nonzero(sel)[0]
        o1 = torch.empty((len(rows), H, 512), dtype=torch.bfloat16, device=DEV)
        l1 = torch.empty((len(rows), H), dtype=torch.float32, device=DEV)
        hs.hs_sparse_attn_decode(q[rows].contiguous(), cache, _t(idx[rows]), 0.04, o1, l1)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(o1), _bits(out[rows]))
        assert torch.equal(l1, lse[rows])


def test_mixed_attention_flags_by_row():
    """No row_req: the flags are indexed by row directly."""
    hs = lib()
    g = np.random.default_rng(13)
    R, H, K, NA, NH = 4, 64, 100, 900, 300
    q = _bf16(g.standard_normal((R, H, 576)) / 24).to(DEV)
    kv_a = _bf16(g.standard_normal((NA, 576)) / 24).to(DEV)
    kv_h = _bf16(g.standard_normal((NH, 576)) / 24).to(DEV)
    idx = g.integers(0, NH, size=(R, K)).astype(np.int32)
    flags = np.array([0, 1, 1, 0], np.int32)
    out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((R, H), dtype=torch.float32, device=DEV)
    hs.hs_sparse_attn_decode_mixed(q, kv_a, kv_h, None, _t(flags), _t(idx), 0.04, out, lse)
    ref, ref_lse = O.sparse_attn_decode_mixed(q.cpu(), kv_a.cpu(), kv_h.cpu(), None, flags, idx,
                                              0.04)
    torch.cuda.synchronize()
    check_attn(out, ref, lse, ref_lse)


def test_mixed_attention_unknown_request_gives_empty_row():
    hs = lib()
    g = np.random.default_rng(12)
    R, H, K, N = 3, 16, 40, 100
    q = _bf16(g.standard_normal((R, H, 576)) / 24).to(DEV)
    kv = _bf16(g.standard_normal((N, 576)) / 24).to(DEV)
    idx = g.integers(0, N, size=(R, K)).astype(np.int32)
    req = np.array([0, 5, -1], np.int32)
    fully = np.array([1, 0], np.int32)
    out = torch.full((R, H, 512), 3.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((R, H), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hs.hs_sparse_attn_decode_mixed(q, kv, kv, _t(req), _t(fully), _t(idx), 0.04, out, lse, st)
    ref, ref_lse = O.sparse_attn_decode_mixed(q.cpu(), kv.cpu(), kv.cpu(), req, fully, idx, 0.04)
    torch.cuda.synchronize()
    check_attn(out, ref, lse, ref_lse)
    assert int(st.item()) == O.STATUS_INDEX
    assert (out[1:] == 0).all()


def test_reclaim_flow_resident_to_host_backed():
    """Two requests on the paged resident cache; the pages are backed up to
    the host pool as they are written. A reclaim takes request 0's old pages
    (they are then reused, i.e. overwritten); request 0 is reset in the hot
    buffer and served by swap-in from the host pool, request 1 stays on the
    resident cache, and one mixed launch attends over both. Every row's
    output matches the all-resident step bit for bit and the oracle over the
    logical rows."""
    hs = lib()
    g = np.random.default_rng(21)
    bs, n_step, S, H, K = 16, 2, 256, 128, 96
    L = [517, 300]                                  # committed positions
    B = len(L)
    nblk = [(l + n_step + bs - 1) // bs for l in L]   # blocks incl. step tokens
    stride = max(nblk) + 1
    n_phys = sum(nblk) + 8
    # resident cache: pages in shuffled physical blocks
    perm = g.permutation(n_phys)
    bt = np.full((B, stride), -1, np.int32)
    k = 0
    for b in range(B):
        bt[b, : nblk[b]] = perm[k:k + nblk[b]]
        k += nblk[b]
    kv_res = _bf16(g.standard_normal((n_phys * bs, 576)) / 24).to(DEV)
    # host pool with its own shuffled page table; every page backed up
    hbt = g.permutation(B * stride).reshape(B, stride).astype(np.int32)
    pool = torch.zeros((B * stride * bs, 576), dtype=torch.bfloat16, pin_memory=True)
    src = np.concatenate([bt[b, : nblk[b]] for b in range(B)]).astype(np.int32)
    dst = np.concatenate([hbt[b, : nblk[b]] for b in range(B)]).astype(np.int32)
    hs.hs_backup_pages([kv_res], [pool], _t(src[None]), _t(dst), _t(np.zeros_like(dst)), bs, 1)
    torch.cuda.synchronize()
    # rows: n_step verify rows per request with causal lengths L+1 .. L+n_step
    # (the step tokens at positions L ..), top-k over each row's prefix
    req = np.repeat(np.arange(B, dtype=np.int32), n_step)
    clen = np.array([L[b] + 1 + i for b in range(B) for i in range(n_step)], np.int32)
    R = len(req)
    topk = np.stack([g.choice(c, size=K, replace=False) for c in clen]).astype(np.int32)
    topk[0, -5:] = -1                               # padding
    q = _bf16(g.standard_normal((R, H, 576)) / 24).to(DEV)
    scale = 0.04

    # step 1: both requests fully resident
    idx1 = torch.empty((R, K), dtype=torch.int32, device=DEV)
    hs.hs_resolve_topk(_t(req), _t(clen), _t(bt), _t(topk), bs, bs, idx1)
    out1 = torch.empty((R, H, 512), dtype=torch.bfloat16, device=DEV)
    lse1 = torch.empty((R, H), dtype=torch.float32, device=DEV)
    hs.hs_sparse_attn_decode(q, kv_res, idx1, scale, out1, lse1)

    # reclaim: request 0's old pages go (scan order takes request 0 first)
    d_bt = _t(bt)
    need = nblk[0] - 2
    freed = torch.empty(need, dtype=torch.int32, device=DEV)
    fully = torch.empty(B, dtype=torch.int32, device=DEV)
    hs.hs_reclaim_resident(d_bt, _t(np.asarray(nblk, np.int32)), need, freed, fully)
    torch.cuda.synchronize()
    assert np_(fully).tolist() == [0, 1]
    assert sorted(np_(freed).tolist()) == sorted(bt[0, :need].tolist())
    kv_before = kv_res.cpu()
    for blk in np_(freed).tolist():                 # the pages are reused
        kv_res[blk * bs:(blk + 1) * bs] = _bf16(g.standard_normal((bs, 576))).to(DEV)

    # step 2: request 0 through the hot buffer, request 1 still resident
    S_tot = S + n_step
    hot = torch.zeros((B * S_tot, 576), dtype=torch.bfloat16, device=DEV)
    buf = hs.HsBuffer(B, S, n_step, stride * bs, bs, hot, pool, _t(hbt))
    hs.hs_request_reset(buf, 0)
    for i in range(n_step):                         # the step tokens' KV
        t = L[0] + i
        row = int(bt[0, t // bs]) * bs + t % bs     # still-held last blocks
        hot[S + i] = kv_res[row]
    r0 = req == 0
    idx2 = torch.empty((R, K), dtype=torch.int32, device=DEV)
    n0 = int(r0.sum())
    hs.hs_swap_in(buf, _t(req[r0]), _t(clen[r0]), _t(np.asarray(L, np.int32)), _t(topk[r0]),
                  idx2[:n0])
    hs.hs_resolve_topk(_t(req[~r0]), _t(clen[~r0]), d_bt, _t(topk[~r0]), bs, bs, idx2[n0:])
    out2 = torch.full((R, H, 512), 5.0, dtype=torch.bfloat16, device=DEV)
    lse2 = torch.empty((R, H), dtype=torch.float32, device=DEV)
    hs.hs_sparse_attn_decode_mixed(q, kv_res, hot, _t(req), fully, idx2, scale, out2, lse2)
    torch.cuda.synchronize()
    assert hs.hs_get_status(buf) == 0
    assert np.array_equal(_bits(out2), _bits(out1))
    assert torch.equal(lse2, lse1)
    # the resident path could no longer serve request 0
    e_idx, _, _ = O.resolve_topk(req[r0], clen[r0], np_(d_bt), topk[r0], bs, bs)
    assert (e_idx[:, :] == -1).sum() > (topk[r0] == -1).sum()

    # the oracle over the logical rows: position t of request b is row
    # bt[b][t // bs] * bs + t % bs of the resident cache before the reclaim
    lrows = np.full((R, K), -1, np.int64)
    for r in range(R):
        b = int(req[r])
        for j in range(K):
            t = int(topk[r, j])
            if 0 <= t < clen[r]:
                lrows[r, j] = int(bt[b, t // bs]) * bs + t % bs
    ref, ref_lse = O.sparse_attn_decode(q.cpu(), kv_before, lrows, scale)
    check_attn(out2, ref, lse2, ref_lse)
