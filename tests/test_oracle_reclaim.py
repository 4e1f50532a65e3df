"""Pins of the oracle's reclaim of resident pages and of the attention over a
batch that mixes fully-resident and host-backed requests ("vllm 分析(十二)
HiSparse 下篇", reclaim_resident_blocks and the fully_resident flag): hand
examples, invariants and the reduction of the mixed batch to one cache."""
import numpy as np
import torch

from oracle import hs_oracle as O


def _table():
    return np.array([[10, 11, 12, 13, 14, -1],
                     [20, 21, -1, -1, -1, -1],
                     [30, -1, 32, 33, 34, 35]], np.int32)


NB = np.array([5, 2, 6], np.int32)


def test_reclaimable_pages_hand_example():
    # every held page but the last two logical blocks; request 1 has only two
    assert O.reclaimable_pages(_table(), NB) == [(0, 0), (0, 1), (0, 2), (2, 0), (2, 2),
                                                 (2, 3)]


def test_reclaim_hand_example():
    bt, freed, fully, n = O.reclaim_resident(_table(), NB, 4)
    assert n == 4
    assert freed.tolist() == [10, 11, 12, 30]
    assert bt.tolist() == [[-1, -1, -1, 13, 14, -1],
                           [20, 21, -1, -1, -1, -1],
                           [-1, -1, 32, 33, 34, 35]]
    assert fully.tolist() == [0, 1, 0]
    # more than is reclaimable: everything but the last two blocks goes
    bt, freed, fully, n = O.reclaim_resident(_table(), NB, 10)
    assert n == 6
    assert freed.tolist() == [10, 11, 12, 30, 32, 33, -1, -1, -1, -1]
    assert bt[2].tolist() == [-1, -1, -1, -1, 34, 35]
    # nothing asked: the table is unchanged and request 2 (a null entry
    # already) is the only one that is not fully resident
    bt, freed, fully, n = O.reclaim_resident(_table(), NB, 0)
    assert n == 0 and freed.size == 0 and np.array_equal(bt, _table())
    assert fully.tolist() == [1, 1, 0]


def test_reclaim_invariants_random():
    g = np.random.default_rng(5)
    for _ in range(30):
        B, stride = int(g.integers(1, 9)), int(g.integers(1, 12))
        bt = g.permutation(B * stride).reshape(B, stride).astype(np.int32)
        bt[g.random((B, stride)) < 0.15] = -1
        nb = g.integers(-1, stride + 3, size=B).astype(np.int32)
        n_recl = len(O.reclaimable_pages(bt, nb))
        a, c = int(g.integers(0, 8)), int(g.integers(0, 8))
        t1, f1, _, n1 = O.reclaim_resident(bt, nb, a)
        t2, f2, fully2, n2 = O.reclaim_resident(t1, nb, c)
        t3, f3, fully3, n3 = O.reclaim_resident(bt, nb, a + c)
        # two reclaims in a row take what one reclaim of the sum takes
        assert np.array_equal(t2, t3) and np.array_equal(fully2, fully3)
        assert f3[:n3].tolist() == f1[:n1].tolist() + f2[:n2].tolist()
        assert n3 == min(a + c, n_recl)
        # released ids are exactly the entries that turned to -1
        gone = (bt >= 0) & (t3 < 0)
        assert sorted(bt[gone].tolist()) == sorted(f3[:n3].tolist())
        assert (f3[n3:] == -1).all()
        for b in range(B):
            n = min(max(int(nb[b]), 0), stride)
            # the last two logical blocks and blocks past n are never touched
            assert np.array_equal(t3[b, max(n - 2, 0):], bt[b, max(n - 2, 0):])
            assert fully3[b] == int((t3[b, :n] >= 0).all())


def _bf16(a):
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def _mixed_case(seed):
    g = np.random.default_rng(seed)
    R, H, K, NA, NH = 6, 3, 9, 40, 17
    q = _bf16(g.standard_normal((R, H, 576)) / 8)
    kv_a = _bf16(g.standard_normal((NA, 576)) / 8)
    kv_h = _bf16(g.standard_normal((NH, 576)) / 8)
    idx = g.integers(-2, NA + 2, size=(R, K)).astype(np.int32)
    req = np.array([0, 1, 1, 2, 0, 2], np.int32)
    fully = np.array([1, 0, 1], np.int32)
    return q, kv_a, kv_h, idx, req, fully


def test_mixed_batch_reduces_to_one_cache():
    """Stacking the hot cache under the resident one and shifting the hot rows'
    valid indices by the resident row count gives the same attention."""
    q, kv_a, kv_h, idx, req, fully = _mixed_case(1)
    out, lse = O.sparse_attn_decode_mixed(q, kv_a, kv_h, req, fully, idx, 0.3)
    NA, NH = kv_a.shape[0], kv_h.shape[0]
    idx2 = idx.copy()
    for r in range(idx.shape[0]):
        if fully[req[r]] == 0:
            ok = (idx[r] >= 0) & (idx[r] < NH)
            idx2[r] = np.where(ok, idx[r] + NA, -1)
        else:
            idx2[r] = np.where((idx[r] >= 0) & (idx[r] < NA), idx[r], -1)
    ref, ref_lse = O.sparse_attn_decode(q, torch.cat([kv_a, kv_h]), idx2, 0.3)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = ~np.isneginf(ref_lse)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-12)
    # an index valid in the resident cache but past the hot one is skipped
    assert any(fully[req[r]] == 0 and (idx[r] >= NH).any() and (idx[r] < NA).any()
               for r in range(idx.shape[0]))


def test_mixed_batch_rows_ignore_the_other_cache():
    q, kv_a, kv_h, idx, req, fully = _mixed_case(2)
    out, _ = O.sparse_attn_decode_mixed(q, kv_a, kv_h, req, fully, idx, 0.3)
    out_a, _ = O.sparse_attn_decode_mixed(q, kv_a, kv_h * 3, req, fully, idx, 0.3)
    out_h, _ = O.sparse_attn_decode_mixed(q, kv_a * 3, kv_h, req, fully, idx, 0.3)
    res = fully[req] != 0
    np.testing.assert_array_equal(out[res], out_a[res])
    np.testing.assert_array_equal(out[~res], out_h[~res])
    assert not np.allclose(out[res], out_h[res])


def test_mixed_batch_unknown_request_and_no_flags():
    q, kv_a, kv_h, idx, req, fully = _mixed_case(3)
    req = req.copy()
    req[2] = 7
    out, lse = O.sparse_attn_decode_mixed(q, kv_a, kv_h, req, fully, idx, 0.3)
    assert (out[2] == 0).all() and np.isneginf(lse[2]).all()
    # no flags: every row reads the resident cache, as sparse_attn_decode
    out0, lse0 = O.sparse_attn_decode_mixed(q, kv_a, kv_h, None, None, idx, 0.3)
    ref, ref_lse = O.sparse_attn_decode(q, kv_a, idx, 0.3)
    np.testing.assert_array_equal(out0, ref)
    np.testing.assert_array_equal(lse0, ref_lse)
