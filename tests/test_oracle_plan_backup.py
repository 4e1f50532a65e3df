"""CPU pins of the oracle's next-row functions: the leader/follower swap plan
and the page backup ("vllm 分析(十二) HiSparse 下篇", resolve_topk's
apply_plan and section 数据 back up)."""
import numpy as np

from oracle import hs_oracle as O


def _rows(n, base):
    # distinct recognisable rows: row i is filled with base + i
    return (np.arange(n, dtype=np.uint16)[:, None] + np.uint16(base)) * np.ones((1, 576), np.uint16)


def test_backup_pages_hand_example():
    # two layers, block_rows 2, blocks_per_kv_block 3; one transfer of layer
    # blocks (4, 1) to host block 2, page offset 1 -> host page 7 -> rows 14, 15
    src = [_rows(10, 100), _rows(10, 200)]
    dst = [np.zeros((20, 576), np.uint16), np.zeros((20, 576), np.uint16)]
    O.backup_pages(src, dst, src_blocks=[[4], [1]], dst_blocks=[2], page_offsets=[1],
                   blocks_per_kv_block=3, block_rows=2)
    assert (dst[0][14] == 108).all() and (dst[0][15] == 109).all()   # rows 8, 9 of layer 0
    assert (dst[1][14] == 202).all() and (dst[1][15] == 203).all()   # rows 2, 3 of layer 1
    untouched = [r for r in range(20) if r not in (14, 15)]
    assert (dst[0][untouched] == 0).all() and (dst[1][untouched] == 0).all()


def test_backup_pages_two_transfers_distinct_pages():
    src = [_rows(12, 10)]
    dst = [np.zeros((26, 576), np.uint16)]
    O.backup_pages(src, dst, src_blocks=[[0, 5]], dst_blocks=[0, 3], page_offsets=[2, 0],
                   blocks_per_kv_block=4, block_rows=2)
    # transfer 0: rows 0, 1 -> host page 0*4 + 2 = 2 -> rows 4, 5
    assert (dst[0][4] == 10).all() and (dst[0][5] == 11).all()
    # transfer 1: rows 10, 11 -> host page 3*4 + 0 = 12 -> rows 24, 25
    assert (dst[0][24] == 20).all() and (dst[0][25] == 21).all()
    assert (dst[0][[0, 1, 2, 3, 6, 12, 23]] == 0).all()


def _leader_and_pools():
    # one request, S = 2 slots, 1 step slot, positions 0..5, block 2, host
    # block table [1, 0, 2] (position t -> host row hbt[t // 2] * 2 + t % 2)
    hbt = [[1, 0, 2]]
    leader_pool = _rows(6, 1000)
    buf = O.HotBuffer(1, 2, 1, 6, 2, hbt, leader_pool)
    follower_pool = _rows(6, 5000)
    follower_hot = np.zeros((buf.S_tot, 576), np.uint16)
    return buf, hbt, follower_pool, follower_hot


def test_apply_plan_hand_example():
    buf, hbt, fpool, fhot = _leader_and_pools()
    # positions 0 and 3 needed (L = 6): both miss; victims are slots 0, 1
    buf.swap_in([0], [7], [6], [[3, 0]])
    assert sorted(buf.last_plan) == [(0, 0, 0), (0, 1, 3)]
    O.apply_plan(buf.last_plan, fhot, fpool, hbt, 2, buf.S_tot)
    # position 0 -> host row hbt[0]*2 + 0 = 2; position 3 -> hbt[1]*2 + 1 = 1
    assert (fhot[0] == 5002).all() and (fhot[1] == 5001).all()
    # a hit makes no copy; the next miss takes the older slot
    buf.swap_in([0], [7], [6], [[3, 4]])
    assert buf.last_plan == [(0, 0, 4)]
    O.apply_plan(buf.last_plan, fhot, fpool, hbt, 2, buf.S_tot, row_offset=0)
    assert (fhot[0] == 5004).all() and (fhot[1] == 5001).all()   # position 4 -> row 2*2 + 0


def test_apply_plan_keeps_follower_in_step_with_leader():
    # over a random sequence every resident slot of the follower holds the
    # follower pool's row of the slot's position (the leader's own invariant)
    g = np.random.default_rng(5)
    S, ctx, bs = 4, 16, 4
    hbt = [list(g.permutation(4))]
    buf = O.HotBuffer(1, S, 1, ctx, bs, hbt, _rows(16, 0))
    fpool = _rows(16, 300)
    fhot = np.zeros((buf.S_tot + 3, 576), np.uint16)
    for _ in range(12):
        t = g.choice(ctx, size=3, replace=False)
        buf.swap_in([0], [ctx + 1], [ctx], [list(t)])
        O.apply_plan(buf.last_plan, fhot, fpool, hbt, bs, buf.S_tot, row_offset=3)
        for s in range(S):
            pos = buf.slot_token[0][s]
            if pos >= 0:
                assert (fhot[3 + s] == fpool[O.host_row(np.array(hbt), 0, pos, bs)]).all()
