"""Pins of the oracle's fully-resident index conversion (resolve_topk of
"vllm 分析(十二) HiSparse 下篇", HiSparseCacheHandle.resolve_topk)."""
import json
import os

import numpy as np

from oracle import hs_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLD, "resolve_hand.json")))
    for case in g["cases"]:
        idx, valid, status = O.resolve_topk(
            g["req_id_per_row"], g["row_causal_len"], np.array(g["block_table"]),
            np.array(g["topk"]), g["block_size"], case["phys_block_stride"])
        assert idx.tolist() == case["expected_idx"]
        assert valid.tolist() == case["expected_valid"]
        assert status == case["expected_status"]


def test_identity_table_is_identity():
    # block table b -> consecutive blocks starting at 0 with stride == bs:
    # the physical row is the position itself.
    bs, nblk = 8, 6
    bt = np.arange(nblk)[None, :]
    topk = np.array([[0, 7, 8, 47, 13, -1]])
    idx, valid, st = O.resolve_topk([0], [48], bt, topk, bs, bs)
    assert idx.tolist() == [[0, 7, 8, 47, 13, -1]]
    assert valid.tolist() == [5] and st == 0


def test_round_trip_recovers_block_and_offset():
    rng = np.random.default_rng(11)
    bs, nblk, B = 16, 9, 3
    perm = rng.permutation(B * nblk).reshape(B, nblk)
    req = np.array([0, 2, 1, 2])
    clen = np.array([nblk * bs] * 4)
    topk = rng.integers(0, nblk * bs, size=(4, 20))
    idx, valid, st = O.resolve_topk(req, clen, perm, topk, bs, bs)
    assert st == 0 and valid.tolist() == [20] * 4
    for r in range(4):
        for j in range(20):
            t = topk[r, j]
            assert idx[r, j] // bs == perm[req[r], t // bs]
            assert idx[r, j] % bs == t % bs


def test_errors_and_padding():
    bt = np.array([[0, -1]])
    # t = 5 falls in an unallocated block; t = 9 is beyond the causal length
    idx, valid, st = O.resolve_topk([0], [8], bt, np.array([[1, 5, 9, -3]]), 4, 4)
    assert idx.tolist() == [[1, -1, -1, -1]]
    assert valid.tolist() == [1]
    assert st == O.STATUS_INDEX
