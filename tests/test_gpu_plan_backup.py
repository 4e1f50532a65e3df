"""GPU parity of the next rows: a swap plan repeated for follower caches
(hs_swap_apply_plan) and the page backup of several layers (hs_backup_pages),
bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import hs_oracle as O
from gpu_util import lib, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a):
    return torch.as_tensor(np.ascontiguousarray(a), device=DEV)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("seed", range(3))
def test_apply_plan_followers_track_leader(seed):
    hs = lib()
    g = np.random.default_rng(77 + seed)
    B, S, n_step, bs, max_ctx = 3, 6, 2, 4, 40
    nblk = max_ctx // bs
    S_tot = S + n_step
    hbt = g.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    pool = W.host_pool_tensor(B * nblk * bs, seed, device=DEV)
    hot = torch.zeros((B * S_tot, 576), dtype=torch.bfloat16, device=DEV)
    buf = hs.HsBuffer(B, S, n_step, max_ctx, bs, hot, pool, _t(hbt))
    ref = O.HotBuffer(B, S, n_step, max_ctx, bs, hbt, pool.clone())
    # two followers: the second one's rows start at an offset in a larger cache
    offs = [0, 5]
    f_pools = [W.host_pool_tensor(B * nblk * bs, 500 + seed + i, device=DEV) for i in range(2)]
    f_hot = [torch.zeros((offs[i] + B * S_tot + 3, 576), dtype=torch.bfloat16, device=DEV)
             for i in range(2)]
    e_hot = [np.zeros((offs[i] + B * S_tot + 3, 576), np.uint16) for i in range(2)]
    f_pool_bits = [_bits(p) for p in f_pools]
    L = [int(x) for x in g.integers(8, 36, size=B)]
    for call in range(8):
        R = int(g.integers(1, 5))
        req = g.integers(0, B, size=R).astype(np.int32)
        K = int(g.integers(1, 6))
        clen = np.array([L[b] + 1 for b in req], np.int32)
        topk = np.stack([g.integers(0, c, size=K) for c in clen]).astype(np.int32)
        out = torch.empty((R, K), dtype=torch.int32, device=DEV)
        hs.hs_swap_in(buf, _t(req), _t(clen), _t(np.asarray(L, np.int32)), _t(topk), out)
        e_out, _, _, _ = ref.swap_in(req, clen, L, topk)
        assert np.array_equal(np_(out), e_out)
        for i in range(2):
            hs.hs_swap_apply_plan(buf, [f_hot[i]], [f_pools[i]], row_offset=offs[i])
            O.apply_plan(ref.last_plan, e_hot[i], f_pool_bits[i], hbt, bs, S_tot, row_offset=offs[i])
        torch.cuda.synchronize()
        for i in range(2):
            assert np.array_equal(_bits(f_hot[i]), e_hot[i])


def test_apply_plan_many_layers_one_call():
    hs = lib()
    g = np.random.default_rng(3)
    B, S, n_step, bs, max_ctx = 4, 16, 1, 8, 96
    nblk = max_ctx // bs
    S_tot = S + n_step
    hbt = g.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    pool = W.host_pool_tensor(B * nblk * bs, 1, device=DEV)
    hot = torch.zeros((B * S_tot, 576), dtype=torch.bfloat16, device=DEV)
    buf = hs.HsBuffer(B, S, n_step, max_ctx, bs, hot, pool, _t(hbt))
    ref = O.HotBuffer(B, S, n_step, max_ctx, bs, hbt, pool.clone())
    n = 5
    f_pools = [W.host_pool_tensor(B * nblk * bs, 40 + i, device=DEV) for i in range(n)]
    f_hot = [torch.zeros((B * S_tot, 576), dtype=torch.bfloat16, device=DEV) for _ in range(n)]
    e_hot = [np.zeros((B * S_tot, 576), np.uint16) for _ in range(n)]
    L = [90] * B
    for call in range(3):
        req = np.arange(B, dtype=np.int32)
        clen = np.array([91] * B, np.int32)
        topk = np.stack([g.choice(90, size=12, replace=False) for _ in range(B)]).astype(np.int32)
        out = torch.empty((B, 12), dtype=torch.int32, device=DEV)
        hs.hs_swap_in(buf, _t(req), _t(clen), _t(np.asarray(L, np.int32)), _t(topk), out)
        ref.swap_in(req, clen, L, topk)
        hs.hs_swap_apply_plan(buf, f_hot, f_pools)
        for i in range(n):
            O.apply_plan(ref.last_plan, e_hot[i], _bits(f_pools[i]), hbt, bs, S_tot)
    torch.cuda.synchronize()
    for i in range(n):
        assert np.array_equal(_bits(f_hot[i]), e_hot[i])


@pytest.mark.parametrize("row_elems", [576, 128])
def test_backup_pages_matches_oracle(row_elems):
    hs = lib()
    g = np.random.default_rng(row_elems)
    n_layers, src_rows, dst_rows, block_rows, bpkb, nt = 3, 240, 480, 4, 3, 25
    src = [torch.randn((src_rows, row_elems), device=DEV).to(torch.bfloat16) for _ in range(n_layers)]
    dst = [torch.zeros((dst_rows, row_elems), dtype=torch.bfloat16).pin_memory()
           for _ in range(n_layers)]
    src_blocks = g.integers(0, src_rows // block_rows, size=(n_layers, nt)).astype(np.int32)
    dst_blocks = g.permutation(dst_rows // (block_rows * bpkb))[:nt].astype(np.int32)
    page_offsets = g.integers(0, bpkb, size=nt).astype(np.int32)
    src_blocks[1, 4] = -1                       # an invalid source block: skipped
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hs.hs_backup_pages(src, dst, _t(src_blocks), _t(dst_blocks), _t(page_offsets), block_rows,
                       bpkb, status=st)
    torch.cuda.synchronize()
    e_src = [_bits(s) for s in src]
    e_dst = [np.zeros((dst_rows, row_elems), np.uint16) for _ in range(n_layers)]
    ok_blocks = src_blocks.copy()
    O.backup_pages(e_src, e_dst, np.where(ok_blocks < 0, 0, ok_blocks), dst_blocks, page_offsets,
                   bpkb, block_rows)
    # the skipped transfer's rows stay untouched in layer 1
    page = int(dst_blocks[4]) * bpkb + int(page_offsets[4])
    e_dst[1][page * block_rows:(page + 1) * block_rows] = 0
    for l in range(n_layers):
        assert np.array_equal(dst[l].view(torch.int16).numpy().view(np.uint16), e_dst[l])
    assert int(st.item()) == O.STATUS_INDEX
