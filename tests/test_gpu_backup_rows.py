"""GPU parity of next row 4 ("vllm 分析(十二) HiSparse 下篇", section c4a kv
cache 写入): row backup by slot mapping, the indexer cache's backup to its
compressed host slots, and follower caches of other row formats (FP8-sized
and indexer-sized rows) repeating a swap plan, all bit-exact against the
oracle, on both the 16-byte and the 4-byte copy paths."""
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


def _rand_bytes(g, rows, width):
    return torch.as_tensor(g.integers(0, 256, size=(rows, width), dtype=np.uint8))


def _offset_view(rows, width, offset, pin):
    """A contiguous [rows][width] uint8 view starting `offset` bytes into its
    allocation (so that only the 4-byte copy path applies)."""
    base = torch.zeros(offset + rows * width, dtype=torch.uint8,
                       pin_memory=pin, device="cpu" if pin else DEV)
    return base[offset:].view(rows, width)


@pytest.mark.parametrize("width,offset", [(1152, 0), (256, 0), (132, 0), (656, 4)])
def test_backup_rows_matches_oracle(width, offset):
    hs = lib()
    g = np.random.default_rng(width + offset)
    n_src, n_dst, n, layers = 700, 900, 400, 3
    src = [_rand_bytes(g, n_src, width).to(DEV) for _ in range(layers)]
    dst = [_offset_view(n_dst, width, offset, pin=True) for _ in range(layers)]
    src_slots = g.integers(-1, n_src, size=n).astype(np.int32)
    dst_slots = g.permutation(n_dst)[:n].astype(np.int32)
    dst_slots[::17] = -1
    src_slots[5] = n_src + 3                       # out of range: skipped, reported
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hs.hs_backup_rows(src, dst, _t(src_slots), _t(dst_slots), st)
    e_dst = [np.zeros((n_dst, width), np.uint8) for _ in range(layers)]
    e_st = O.backup_rows([s.cpu().numpy() for s in src], e_dst, src_slots, dst_slots)
    torch.cuda.synchronize()
    assert int(st.item()) == e_st == O.STATUS_INDEX
    for l in range(layers):
        assert np.array_equal(dst[l].numpy(), e_dst[l])


@pytest.mark.parametrize("sbs,ratio,width", [(16, 4, 132), (64, 4, 256), (8, 1, 144)])
def test_backup_indexer_matches_oracle(sbs, ratio, width):
    hs = lib()
    g = np.random.default_rng(sbs * ratio + width)
    lbs = sbs * ratio
    B, nblk = 3, 6
    host_bt = g.permutation(B * nblk + 4)[:B * nblk].reshape(B, nblk)
    n_dev = B * nblk * sbs + 10
    src = [_rand_bytes(g, n_dev, width).to(DEV)]
    host = [torch.zeros(int(host_bt.max() + 1) * sbs, width, dtype=torch.uint8,
                         pin_memory=True)]
    # a prefill of each request's first L tokens: the compressor wrote one
    # entry per `ratio` tokens (at the group's last token) into device rows
    src_slots, host_slots, pos = [], [], []
    free = list(g.permutation(n_dev))
    for b in range(B):
        L = int(g.integers(lbs, nblk * lbs + 1))
        for p in range(L):
            host_slots.append(int(host_bt[b, p // lbs]) * lbs + p % lbs)
            pos.append(p)
            src_slots.append(int(free.pop()) if p % ratio == ratio - 1 else -1)
    src_slots, host_slots, pos = (np.asarray(x, np.int32) for x in (src_slots, host_slots, pos))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hs.hs_backup_indexer(src, host, _t(src_slots), _t(host_slots), _t(pos), sbs, ratio, st)
    e_host = [np.zeros(tuple(host[0].shape), np.uint8)]
    dst = O.compress_slot_mapping(host_slots, pos, sbs, ratio)
    e_st = O.backup_rows([src[0].cpu().numpy()], e_host, src_slots, dst)
    torch.cuda.synchronize()
    assert int(st.item()) == e_st == 0
    assert np.array_equal(host[0].numpy(), e_host[0])


def test_apply_plan_other_row_formats():
    """Followers of other row sizes (an FP8-sized 656-byte row, a 132-byte
    indexer-sized row, one view 4 bytes off alignment) repeat the plan."""
    hs = lib()
    g = np.random.default_rng(9)
    B, S, n_step, bs, max_ctx = 4, 12, 2, 8, 80
    nblk = max_ctx // bs
    S_tot = S + n_step
    hbt = g.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    pool = W.host_pool_tensor(B * nblk * bs, 4, device=DEV)
    hot = torch.zeros((B * S_tot, 576), dtype=torch.bfloat16, device=DEV)
    buf = hs.HsBuffer(B, S, n_step, max_ctx, bs, hot, pool, _t(hbt))
    ref = O.HotBuffer(B, S, n_step, max_ctx, bs, hbt, pool.clone())
    fmts = [(656, 0), (132, 0), (656, 4)]
    f_pool, f_hot, e_hot = [], [], []
    for width, off in fmts:
        p = _offset_view(B * nblk * bs, width, off, pin=True)
        p.copy_(_rand_bytes(g, B * nblk * bs, width))
        f_pool.append(p)
        f_hot.append(_offset_view(B * S_tot, width, off, pin=False))
        e_hot.append(np.zeros((B * S_tot, width), np.uint8))
    L = [int(x) for x in g.integers(20, max_ctx - n_step, size=B)]
    for call in range(6):
        R = int(g.integers(1, 6))
        req = g.integers(0, B, size=R).astype(np.int32)
        K = int(g.integers(1, 9))
        clen = np.array([L[b] + 1 for b in req], np.int32)
        topk = np.stack([g.integers(0, c, size=K) for c in clen]).astype(np.int32)
        out = torch.empty((R, K), dtype=torch.int32, device=DEV)
        hs.hs_swap_in(buf, _t(req), _t(clen), _t(np.asarray(L, np.int32)), _t(topk), out)
        e_out, _, _, _ = ref.swap_in(req, clen, L, topk)
        assert np.array_equal(np_(out), e_out)
        for i in range(len(fmts)):                 # one call per row format
            hs.hs_swap_apply_plan(buf, [f_hot[i]], [f_pool[i]])
        for i in range(len(fmts)):
            O.apply_plan(ref.last_plan, e_hot[i], f_pool[i].numpy(), hbt, bs, S_tot)
        torch.cuda.synchronize()
        for i in range(len(fmts)):
            assert np.array_equal(f_hot[i].cpu().numpy(), e_hot[i]), fmts[i]


def test_backup_rows_and_apply_plan_64_layers():
    """The most layers one call takes (64), for both calls."""
    hs = lib()
    g = np.random.default_rng(64)
    n_l, n_src, n = 64, 50, 30
    src = [_rand_bytes(g, n_src, 144).to(DEV) for _ in range(n_l)]
    dst = [torch.zeros((40, 144), dtype=torch.uint8, pin_memory=True) for _ in range(n_l)]
    ss = g.integers(0, n_src, size=n).astype(np.int32)
    ds = g.permutation(40)[:n].astype(np.int32)
    hs.hs_backup_rows(src, dst, _t(ss), _t(ds))
    e_dst = [np.zeros((40, 144), np.uint8) for _ in range(n_l)]
    O.backup_rows([x.cpu().numpy() for x in src], e_dst, ss, ds)
    torch.cuda.synchronize()
    for l in range(n_l):
        assert np.array_equal(dst[l].numpy(), e_dst[l])
    # follower caches: 64 layers of 16-byte rows on one plan
    B, S, n_step, bs, max_ctx = 2, 4, 1, 4, 16
    nblk = max_ctx // bs
    S_tot = S + n_step
    hbt = g.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    pool = W.host_pool_tensor(B * nblk * bs, 8, device=DEV)
    hot = torch.zeros((B * S_tot, 576), dtype=torch.bfloat16, device=DEV)
    buf = hs.HsBuffer(B, S, n_step, max_ctx, bs, hot, pool, _t(hbt))
    ref = O.HotBuffer(B, S, n_step, max_ctx, bs, hbt, pool.clone())
    f_pool = [_rand_bytes(g, B * nblk * bs, 16).pin_memory() for _ in range(n_l)]
    f_hot = [torch.zeros((B * S_tot, 16), dtype=torch.uint8, device=DEV) for _ in range(n_l)]
    req = np.array([0, 1], np.int32)
    clen = np.array([12, 9], np.int32)
    topk = np.array([[0, 5, 11], [1, 2, 8]], np.int32)
    out = torch.empty((2, 3), dtype=torch.int32, device=DEV)
    hs.hs_swap_in(buf, _t(req), _t(clen), _t(np.array([12, 9], np.int32)), _t(topk), out)
    ref.swap_in(req, clen, [12, 9], topk)
    hs.hs_swap_apply_plan(buf, f_hot, f_pool)
    torch.cuda.synchronize()
    for l in range(n_l):
        e = np.zeros((B * S_tot, 16), np.uint8)
        O.apply_plan(ref.last_plan, e, f_pool[l].numpy(), hbt, bs, S_tot)
        assert np.array_equal(f_hot[l].cpu().numpy(), e)


@pytest.mark.parametrize("width,offset", [(4, 0), (20, 0), (132, 4), (128, 8), (252, 0)])
@pytest.mark.parametrize("pattern", ["blocks", "scattered"])
def test_backup_rows_short_rows_runs(width, offset, pattern):
    """Rows that do not go 16 bytes at a time and are shorter than 256 bytes:
    host rows in runs of consecutive slots (whole and partial blocks, holes,
    entries without a row) or scattered, 2 layers, bit-exact."""
    hs = lib()
    g = np.random.default_rng(width * 7 + offset + (pattern == "blocks"))
    n_src, n_dst, n, layers = 600, 1400, 1000, 2
    src = [_rand_bytes(g, n_src, width).to(DEV) for _ in range(layers)]
    dst = [_offset_view(n_dst, width, offset, pin=True) for _ in range(layers)]
    src_slots = g.integers(0, n_src, size=n).astype(np.int32)
    if pattern == "blocks":
        # blocks of 16 host rows in shuffled order, some cut short
        order = g.permutation(n_dst // 16)
        dst_slots = np.concatenate([b * 16 + np.arange(16) for b in order])[:n].astype(np.int32)
        dst_slots[g.integers(0, n, size=40)] = -1
        src_slots[g.integers(0, n, size=40)] = -1
    else:
        dst_slots = g.permutation(n_dst)[:n].astype(np.int32)
        dst_slots[::13] = -1
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hs.hs_backup_rows(src, dst, _t(src_slots), _t(dst_slots), st)
    e_dst = [np.zeros((n_dst, width), np.uint8) for _ in range(layers)]
    e_st = O.backup_rows([s.cpu().numpy() for s in src], e_dst, src_slots, dst_slots)
    torch.cuda.synchronize()
    assert int(st.item()) == e_st == 0
    for l in range(layers):
        assert np.array_equal(dst[l].numpy(), e_dst[l])
