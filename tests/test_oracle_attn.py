"""Pins of the oracle's sparse attention (per row and head, softmax over the
selected 576-dim latent rows, values = the first 512 dims): a pure-Python
brute force on tiny inputs, closed forms and special cases."""
import math

import numpy as np
import pytest
import torch

from oracle import hs_oracle as O

D, DV = O.LATENT_DIM, O.VALUE_DIM


def _bf16(x):
    return torch.tensor(np.asarray(x), dtype=torch.float32).to(torch.bfloat16)


def _brute(qh_list, kv_rows, scale):
    """Brute force with math.fsum / math.exp on Python floats."""
    outs, lses = [], []
    for qh in qh_list:
        s = [scale * math.fsum(a * b for a, b in zip(qh, k)) for k in kv_rows]
        if not s:
            outs.append([0.0] * DV)
            lses.append(-math.inf)
            continue
        m = max(s)
        w = [math.exp(x - m) for x in s]
        tot = math.fsum(w)
        outs.append([math.fsum(w[j] * kv_rows[j][c] for j in range(len(w))) / tot
                     for c in range(DV)])
        lses.append(m + math.log(tot))
    return outs, lses


@pytest.mark.parametrize("seed", range(3))
def test_bruteforce_tiny(seed):
    g = np.random.default_rng(seed)
    R, H, N, K = 2, 2, 9, 5
    q = _bf16(g.standard_normal((R, H, D)))
    kv = _bf16(g.standard_normal((N, D)))
    idx = np.array([[3, -1, 0, 8, 3], [7, 2, -1, -1, 11]])   # 11 >= N is skipped
    scale = 0.05
    out, lse = O.sparse_attn_decode(q, kv, idx, scale)
    qf, kvf = q.double().numpy(), kv.double().numpy()
    for r in range(R):
        rows = [kvf[j].tolist() for j in idx[r] if 0 <= j < N]
        bo, bl = _brute([qf[r, h].tolist() for h in range(H)], rows, scale)
        assert np.allclose(out[r], np.array(bo), rtol=1e-12, atol=1e-14)
        assert np.allclose(lse[r], np.array(bl), rtol=1e-12)


def test_single_valid_row_returns_its_value_exactly():
    g = np.random.default_rng(1)
    q = _bf16(g.standard_normal((1, 3, D)))
    kv = _bf16(g.standard_normal((4, D)))
    out, lse = O.sparse_attn_decode(q, kv, np.array([[-1, 2, -1]]), 0.1)
    v = kv.double().numpy()[2]
    assert np.array_equal(out[0], np.tile(v[:DV], (3, 1)))
    s = 0.1 * (q.double().numpy()[0] @ v)
    assert np.allclose(lse[0], s, rtol=1e-14)


def test_identical_keys_give_that_value():
    g = np.random.default_rng(2)
    q = _bf16(g.standard_normal((1, 2, D)))
    row = g.standard_normal(D)
    kv = _bf16(np.stack([row] * 5))
    out, lse = O.sparse_attn_decode(q, kv, np.array([[0, 1, 2, 3, 4]]), 0.3)
    v = kv.double().numpy()[0]
    assert np.allclose(out[0], np.tile(v[:DV], (2, 1)), rtol=1e-14, atol=0)
    s = 0.3 * (q.double().numpy()[0] @ v)
    assert np.allclose(lse[0], s + math.log(5), rtol=1e-13)


def test_two_keys_closed_form():
    # q = e_0, k_a = a * e_0 + v_a, k_b = b * e_0 + v_b with values disjoint
    # from dim 0: weights are the logistic function of scale * (a - b).
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 1.0
    kv = np.zeros((2, D))
    kv[0, 0], kv[1, 0] = 2.0, -1.0
    kv[0, 5], kv[1, 7] = 1.5, -0.75
    scale = 0.7
    out, lse = O.sparse_attn_decode(_bf16(q), _bf16(kv), np.array([[0, 1]]), scale)
    pa = 1.0 / (1.0 + math.exp(-scale * 3.0))
    exp = np.zeros(DV); exp[0] = pa * 2.0 + (1 - pa) * -1.0
    exp[5], exp[7] = pa * 1.5, (1 - pa) * -0.75
    assert np.allclose(out[0, 0], exp, rtol=1e-14, atol=1e-15)
    assert math.isclose(lse[0, 0], math.log(math.exp(1.4) + math.exp(-0.7)), rel_tol=1e-14)


def test_value_is_first_512_dims_only():
    # A key whose dims 512..575 are large: they enter the logit but never the
    # output.
    q = np.zeros((1, 1, D)); q[0, 0, 600 - 64] = 1.0    # dim 536 (a rope dim)
    kv = np.zeros((1, D)); kv[0, 536] = 4.0; kv[0, 3] = 0.5
    out, lse = O.sparse_attn_decode(_bf16(q), _bf16(kv), np.array([[0]]), 1.0)
    assert out.shape == (1, 1, DV)
    exp = np.zeros(DV); exp[3] = 0.5
    assert np.array_equal(out[0, 0], exp)
    assert lse[0, 0] == 4.0


def test_duplicate_entry_counts_twice():
    # listing key a twice equals one key a with its logit raised by ln 2
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 1.0
    kv = np.zeros((2, D)); kv[0, 0] = 1.0; kv[1, 0] = 0.0
    kv[0, 9] = 1.0; kv[1, 10] = 1.0
    out, _ = O.sparse_attn_decode(_bf16(q), _bf16(kv), np.array([[0, 0, 1]]), 1.0)
    wa = 2 * math.e / (2 * math.e + 1)
    assert math.isclose(out[0, 0, 9], wa, rel_tol=1e-14)
    assert math.isclose(out[0, 0, 10], 1 - wa, rel_tol=1e-14)


def test_planted_dominant_key():
    g = np.random.default_rng(4)
    q = g.standard_normal((1, 1, D)) / 24
    kv = g.standard_normal((64, D)) / 24
    q[0, 0, :] = 0; q[0, 0, 0] = 1.0
    kv[:, 0] = 0; kv[17, 0] = 60.0            # logit 60 above every other
    out, _ = O.sparse_attn_decode(_bf16(q), _bf16(kv), np.arange(64)[None, :], 1.0)
    v = _bf16(kv).double().numpy()[17, :DV]
    assert np.allclose(out[0, 0], v, rtol=0, atol=1e-20)


def test_empty_row_and_permutation_invariance():
    g = np.random.default_rng(6)
    q = _bf16(g.standard_normal((2, 2, D)))
    kv = _bf16(g.standard_normal((6, D)))
    out, lse = O.sparse_attn_decode(q, kv, np.array([[-1, -1, 9], [0, 1, 5]]), 0.05)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    out2, lse2 = O.sparse_attn_decode(q, kv, np.array([[-1, -1, -1], [5, 0, 1]]), 0.05)
    assert np.allclose(out2[1], out[1], rtol=1e-13) and np.allclose(lse2[1], lse[1], rtol=1e-14)


def test_rows_helper_matches_full():
    g = np.random.default_rng(8)
    q = _bf16(g.standard_normal((3, 2, D)))
    kv = _bf16(g.standard_normal((10, D)))
    idx = np.array([[1, 2, 3], [4, -1, 9], [0, 0, 7]])
    out, lse = O.sparse_attn_decode(q, kv, idx, 0.1)
    kvf = kv.double().numpy()
    o2, l2 = O.sparse_attn_decode_rows(q, lambda rows: kvf[rows], idx, 0.1, [0, 2])
    assert np.array_equal(o2[0], out[0]) and np.array_equal(l2[2], lse[2])
