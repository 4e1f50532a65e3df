"""The seeded generators: deterministic, the stated shapes and structure."""
import numpy as np

import workloads as W


def test_deterministic_and_distinct():
    c = W.get_config(1)
    req, ri = W.rows_of(c)
    a = W.topk_independent(c, 0, c.L, req, ri)
    b = W.topk_independent(c, 0, c.L, req, ri)
    assert np.array_equal(a, b) and a.shape == (8, 64)
    clen = W.causal_lengths(c.L, req, ri)
    assert clen.tolist() == [513, 514, 515, 516, 301, 302, 303, 304]
    for r in range(8):
        v = a[r][a[r] >= 0]
        assert len(set(v.tolist())) == len(v) == 64 and v.max() < clen[r]


def test_padding_when_context_short():
    g = W.rng(0, "x")
    out = W.distinct_uniform(g, 5, 8)
    assert sorted(out[:5].tolist()) == [0, 1, 2, 3, 4] and out[5:].tolist() == [-1] * 3


def test_locality_reuse_fraction():
    c = W.get_config(3)
    sets = W.locality_sets(c, 32768, 7, 5)
    for t in range(1, 5):
        prev, cur = set(sets[t - 1].tolist()), set(sets[t].tolist())
        assert len(cur) == 2048
        assert len(prev & cur) == round(0.8 * 2048)
        fresh = cur - prev
        recent = [x for x in fresh if x >= 32768 - 4096]
        assert len(recent) >= len(fresh) // 2


def test_shared_sets_shuffled_per_row():
    c = W.get_config(3)
    c.B = 2
    sets = [W.locality_sets(c, 32768, b, 2) for b in range(2)]
    tk = W.topk_shared_sets(c, sets, 1)
    assert tk.shape == (8, 2048)
    assert sorted(tk[0].tolist()) == sorted(tk[3].tolist()) == sorted(sets[0][1].tolist())
    assert not np.array_equal(tk[0], tk[1])


def test_block_table_is_a_permutation():
    bt, total = W.shuffled_block_table(2, "bt", [3, 2, 4])
    vals = bt[bt >= 0]
    assert total == 9 and sorted(vals.tolist()) == list(range(9))
    assert bt[1, 2:].tolist() == [-1, -1]


def test_planted_logits():
    c = W.get_config(1)
    lg, dr, planted = W.planted_logits(c)
    assert lg.shape == (2, 4, 1024) and dr.shape == (2, 3)
    for b in range(2):
        for i in range(3):
            row = lg[b, i].numpy()
            if planted[b, i]:
                assert row.argmax() == dr[b, i] and (row == row.max()).sum() == 1
            else:
                assert row[dr[b, i]] < row.max()


def test_bf16_normal_scale():
    x = W.bf16_normal((64, 576), W.KV_SCALE, 0, "kv")
    y = W.bf16_normal((64, 576), W.KV_SCALE, 0, "kv")
    assert x.dtype.is_floating_point and (x == y).all()
    assert abs(x.float().std().item() - 1 / 24) < 0.003
