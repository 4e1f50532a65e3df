"""GPU behaviour at the degenerate sizes the calls accept: no rows, rows with
no keys, empty top-k, no drafts, empty copy lists, against the oracle."""
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


def _bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def test_attention_without_keys_and_without_rows():
    hs = lib()
    g = np.random.default_rng(0)
    q = _bf16(g.standard_normal((3, 128, 576)) / 24).to(DEV)
    kv = _bf16(g.standard_normal((10, 576)) / 24).to(DEV)
    idx = torch.empty((3, 0), dtype=torch.int32, device=DEV)
    out = torch.full((3, 128, 512), 9.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros((3, 128), dtype=torch.float32, device=DEV)
    hs.hs_sparse_attn_decode(q, kv, idx, 0.04, out, lse)
    torch.cuda.synchronize()
    assert (out == 0).all() and torch.isneginf(lse).all()
    # no rows: nothing is written
    out0 = torch.empty((0, 128, 512), dtype=torch.bfloat16, device=DEV)
    hs.hs_sparse_attn_decode(q[:0], kv, torch.empty((0, 5), dtype=torch.int32, device=DEV), 0.04,
                             out0)
    torch.cuda.synchronize()


def test_resolve_empty():
    hs = lib()
    bt = _t(np.arange(8, dtype=np.int32).reshape(2, 4))
    out = torch.empty((0, 7), dtype=torch.int32, device=DEV)
    hs.hs_resolve_topk(_t(np.zeros(0, np.int32)), _t(np.zeros(0, np.int32)), bt,
                       torch.empty((0, 7), dtype=torch.int32, device=DEV), 16, 16, out)
    valid = torch.full((2,), 5, dtype=torch.int32, device=DEV)
    out2 = torch.empty((2, 0), dtype=torch.int32, device=DEV)
    hs.hs_resolve_topk(_t(np.array([0, 1], np.int32)), _t(np.array([5, 9], np.int32)), bt,
                       torch.empty((2, 0), dtype=torch.int32, device=DEV), 16, 16, out2, valid)
    torch.cuda.synchronize()
    assert np_(valid).tolist() == [0, 0]


def _small_buffer(hs, g, B=2, S=6, n_step=2, bs=4, max_ctx=24):
    nblk = max_ctx // bs
    hbt = g.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    pool = W.host_pool_tensor(B * nblk * bs, 3, device=DEV)
    hot = torch.zeros((B * (S + n_step), 576), dtype=torch.bfloat16, device=DEV)
    buf = hs.HsBuffer(B, S, n_step, max_ctx, bs, hot, pool, _t(hbt))
    ref = O.HotBuffer(B, S, n_step, max_ctx, bs, hbt, pool.clone())
    return buf, ref, hot, pool, hbt


def test_swap_in_empty_batch_and_empty_topk():
    hs = lib()
    g = np.random.default_rng(1)
    buf, ref, hot, _, _ = _small_buffer(hs, g)
    L = np.array([10, 7], np.int32)
    # no rows at all
    hs.hs_swap_in(buf, _t(np.zeros(0, np.int32)), _t(np.zeros(0, np.int32)), _t(L),
                  torch.empty((0, 3), dtype=torch.int32, device=DEV),
                  torch.empty((0, 3), dtype=torch.int32, device=DEV))
    ref.swap_in(np.zeros(0, np.int32), np.zeros(0, np.int32), L, np.zeros((0, 3), np.int32))
    # rows with only padding
    out = torch.empty((2, 3), dtype=torch.int32, device=DEV)
    valid = torch.empty(2, dtype=torch.int32, device=DEV)
    topk = np.full((2, 3), -1, np.int32)
    hs.hs_swap_in(buf, _t(np.array([0, 1], np.int32)), _t(np.array([11, 8], np.int32)), _t(L),
                  _t(topk), out, valid)
    e_out, e_valid, e_st, _ = ref.swap_in(np.array([0, 1]), np.array([11, 8]), L, topk)
    torch.cuda.synchronize()
    assert np.array_equal(np_(out), e_out) and np.array_equal(np_(valid), e_valid)
    assert hs.hs_get_status(buf) == e_st == 0
    ts, stok, sts = buf.dump()
    for b in range(2):
        assert stok[b].tolist() == ref.slot_token[b]
    assert buf.clock == ref.now
    buf.close()


def test_verify_without_drafts():
    """d = 0: the anchor's argmax is the next token, nothing is accepted, and
    the anchor's KV row is committed."""
    hs = lib()
    g = np.random.default_rng(2)
    buf, ref, hot, pool, hbt = _small_buffer(hs, g, n_step=1)
    L = [10, 7]
    kv_len = _t(np.asarray(L, np.int32))
    logits = torch.randn((2, 1, 300), generator=torch.Generator().manual_seed(4)).to(DEV)
    skv = _bf16(g.standard_normal((2, 1, 576))).to(DEV)
    acc = torch.empty(2, dtype=torch.int32, device=DEV)
    nxt = torch.empty_like(acc)
    hs.hs_verify_finalize(buf, logits, torch.empty((2, 0), dtype=torch.int32, device=DEV), skv,
                          kv_len, acc, nxt)
    e_acc, e_nxt, e_L, e_st = O.verify_finalize(ref, logits.cpu(), np.zeros((2, 0), np.int32),
                                                skv.cpu(), L)
    torch.cuda.synchronize()
    assert np_(acc).tolist() == list(e_acc) == [0, 0]
    assert np.array_equal(np_(nxt), e_nxt) and np.array_equal(np_(kv_len), e_L)
    assert hs.hs_get_status(buf) == e_st == 0
    assert np.array_equal(pool.view(torch.int16).numpy().view(np.uint16), ref.host_pool)
    buf.close()


def test_empty_copy_calls():
    hs = lib()
    g = np.random.default_rng(3)
    src = [_bf16(g.standard_normal((8, 576))).to(DEV)]
    dst = [torch.zeros((8, 576), dtype=torch.bfloat16, pin_memory=True)]
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    hs.hs_backup_rows(src, dst, e, e)
    hs.hs_backup_indexer(src, dst, e, e, e, 4, 2)
    hs.hs_backup_pages(src, dst, torch.empty((1, 0), dtype=torch.int32, device=DEV), e, e, 4, 1)
    buf, ref, _, _, _ = _small_buffer(hs, g)
    hs.hs_swap_apply_plan(buf, [], [])
    # reclaim with nothing asked for, and over an empty batch
    table = np.array([[1, 2, 3, 4], [5, 6, -1, -1]], np.int32)
    nb = np.array([4, 2], np.int32)
    bt = _t(table)
    fr = _t(np.ones(2, np.int32))
    n_freed = torch.full((1,), 9, dtype=torch.int32, device=DEV)
    hs.hs_reclaim_resident(bt, _t(nb), 0, None, fr, n_freed)
    e_tab, _, e_fr, e_n = O.reclaim_resident(table, nb, 0)
    freed = torch.full((3,), 7, dtype=torch.int32, device=DEV)
    n2 = torch.full((1,), 9, dtype=torch.int32, device=DEV)
    hs.hs_reclaim_resident(torch.empty((0, 4), dtype=torch.int32, device=DEV),
                           torch.empty(0, dtype=torch.int32, device=DEV), 3, freed, None, n2)
    torch.cuda.synchronize()
    assert (dst[0] == 0).all()
    assert np.array_equal(np_(bt), e_tab) and int(n_freed.item()) == e_n == 0
    assert np.array_equal(np_(fr), e_fr) and np_(fr).tolist() == [1, 1]
    assert np_(freed).tolist() == [-1, -1, -1] and int(n2.item()) == 0
    buf.close()
