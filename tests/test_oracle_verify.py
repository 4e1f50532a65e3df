"""Pins of the oracle's greedy verify and commit against the worked example of
"投机解码的 KV 流转：prefill 阶段 DFlash 也要吃下整个 prompt" (sections ④-⑥
and the closing table)."""
import json
import os

import numpy as np

from oracle import hs_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _logits_with_argmax(argmaxes, V, seed=0):
    g = np.random.default_rng(seed)
    lg = g.standard_normal((1, len(argmaxes), V)).astype(np.float32)
    for i, a in enumerate(argmaxes):
        lg[0, i, a] = lg[0, i].max() + 1.0
    return lg


def test_worked_example_cases():
    g = json.load(open(os.path.join(GOLD, "p2_worked_example.json")))
    V, P = g["vocab"], g["prompt_len"]
    bs, max_ctx, S = 4, 16, 6
    for case in g["cases"]:
        e = case["expected"]
        pool = np.zeros((max_ctx, O.LATENT_DIM), dtype=np.uint16)
        buf = O.HotBuffer(1, S, 4, max_ctx, bs, np.arange(max_ctx // bs)[None, :], pool)
        step_kv = (np.arange(4 * O.LATENT_DIM, dtype=np.uint16).reshape(1, 4, -1) + 1)
        lg = _logits_with_argmax(case["target_argmax_per_input"], V)
        acc, nxt, L, st = O.verify_finalize(buf, lg, np.array([g["drafts"]]), step_kv, [P])
        assert st == 0
        assert acc.tolist() == [e["accept_len"]]
        assert nxt.tolist() == [e["next_token"]]
        assert L.tolist() == [e["kv_len_after"]]
        # target KV covers exactly P + the accepted prefix
        held = sorted(t for t in buf.slot_token[0] if t >= 0)
        assert held == e["committed_positions"]
        for t, k in zip(e["committed_positions"], e["committed_step_rows"]):
            s = buf.token_slot[0][t]
            assert np.array_equal(buf.hot[buf.hot_row(0, s)], step_kv[0, k])
            assert np.array_equal(buf.host_pool[O.host_row(buf.hbt, 0, t, bs)], step_kv[0, k])
        # the token chosen last has no KV yet
        for t in e["positions_without_kv"]:
            assert t not in buf.token_slot[0]
            assert not buf.host_pool[O.host_row(buf.hbt, 0, t, bs)].any()
        if "round2_anchor_position" in e:
            # next round: anchor at L, drafts after it; row i's causal length L+i+1
            Lnew = int(L[0])
            assert Lnew == e["round2_anchor_position"]
            assert [Lnew + i for i in (1, 2, 3)] == e["round2_draft_positions"]
            assert [Lnew + i + 1 for i in range(4)] == e["round2_row_causal_lengths"]


def test_argmax_tie_goes_to_lowest_index():
    row = np.array([0.5, 2.0, -1.0, 2.0, 2.0])
    assert O.argmax_lowest(row) == 1
    assert O.greedy_accept([3, 1], [3]) == (1, 1)
    assert O.greedy_accept([1, 1], [3]) == (0, 1)


def test_accept_prefix_stops_at_first_mismatch():
    # a later agreement after a mismatch does not count
    assert O.greedy_accept([5, 9, 7, 2], [5, 8, 7]) == (1, 9)
    assert O.greedy_accept([5, 8, 7, 2], [5, 8, 7]) == (3, 2)


def test_multi_request_commit_and_capacity():
    V, bs, max_ctx = 8, 4, 8
    pool = np.zeros((2 * max_ctx, O.LATENT_DIM), dtype=np.uint16)
    hbt = np.array([[1, 0], [3, 2]])
    buf = O.HotBuffer(2, 4, 3, max_ctx, bs, hbt, pool)
    lg = np.concatenate([_logits_with_argmax([1, 2, 3], V, 1), _logits_with_argmax([1, 2, 3], V, 2)])
    step_kv = np.ones((2, 3, O.LATENT_DIM), dtype=np.uint16)
    # request 1 sits at L = 6: committing 3 rows would pass max_ctx = 8
    acc, nxt, L, st = O.verify_finalize(buf, lg, np.array([[1, 2], [1, 2]]), step_kv, [2, 6])
    assert acc.tolist() == [2, 2] and nxt.tolist() == [3, 3]
    assert L.tolist() == [5, 6]
    assert st == O.STATUS_CAPACITY
    assert sorted(buf.token_slot[0]) == [2, 3, 4] and buf.token_slot[1] == {}
    # host rows of request 0, positions 2..4: block 1 -> host block 0, block 0 -> 1
    assert pool[4 + 2].any() and pool[4 + 3].any() and pool[0].any() and not pool[1].any()
