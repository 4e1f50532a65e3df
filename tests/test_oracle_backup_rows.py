"""Pins of the oracle's row backup and of the indexer cache's compressed host
slots ("vllm 分析(十二) HiSparse 下篇", section c4a kv cache 写入): hand
examples, and the host slots rebuilt by walking the tokens block by block."""
import numpy as np

from oracle import hs_oracle as O


def test_compress_slot_mapping_hand_example():
    # 2 entries per storage block, one entry per 4 tokens: logical blocks of
    # 8 token slots; logical host block 3 holds slots 24..31
    slots = [24, 27, 28, 31, -1, 40, 30]
    pos = [8, 11, 12, 15, 9, 0, -1]
    got = O.compress_slot_mapping(slots, pos, 2, 4).tolist()
    assert got == [6, 6, 7, 7, -1, 10, -1]


def test_compress_slot_mapping_matches_a_block_walk():
    """Walk each request's tokens in order; every compress_ratio tokens close
    one entry, appended to the storage block of their logical block. The
    entry each token falls into must be the mapping's host row."""
    g = np.random.default_rng(3)
    for sbs, ratio in [(1, 1), (2, 4), (16, 4), (8, 128), (64, 1)]:
        lbs = sbs * ratio
        nblk = 5
        host_bt = g.permutation(3 * nblk)[:nblk]          # logical -> host block
        n_tok = nblk * lbs
        pos = np.arange(n_tok)
        slots = host_bt[pos // lbs] * lbs + pos % lbs
        got = O.compress_slot_mapping(slots, pos, sbs, ratio)
        filled = {}                                    # host block -> entries so far
        for p in range(n_tok):
            hb = int(host_bt[p // lbs])
            if p % ratio == 0:                         # a new group opens an entry
                filled[hb] = filled.get(hb, 0) + 1
            assert got[p] == hb * sbs + filled[hb] - 1
        assert all(v == sbs for v in filled.values())  # every block exactly full


def test_backup_rows_hand_example():
    src = [np.arange(15, dtype=np.uint8).reshape(5, 3),
           np.arange(100, 115, dtype=np.uint8).reshape(5, 3)]
    dst = [np.zeros((4, 3), np.uint8), np.zeros((4, 3), np.uint8)]
    st = O.backup_rows(src, dst, [0, 2, -1, 4, 7], [3, 0, 1, -1, 2])
    assert st == O.STATUS_INDEX                        # source row 7 does not exist
    assert dst[0].tolist() == [[6, 7, 8], [0, 0, 0], [0, 0, 0], [0, 1, 2]]
    assert dst[1].tolist() == [[106, 107, 108], [0, 0, 0], [0, 0, 0], [100, 101, 102]]
    assert O.backup_rows(src, dst, [1], [2]) == 0
    assert dst[0][2].tolist() == [3, 4, 5]
