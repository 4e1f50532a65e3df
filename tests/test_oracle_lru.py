"""Pins of the oracle's hot buffer: swap-in and commit against (a) a worked
example done by hand, (b) an independent naive model that selects each victim
by a linear scan, and (c) the invariants the pages state for the core maps
("hiSparse-MTP", core state maps): slots and positions map 1:1, every
requested position is resident after a swap-in, every hot row equals its host
row."""
import json
import os

import numpy as np
import pytest

from oracle import hs_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
D = O.LATENT_DIM


def _pool(rows, seed=0):
    g = np.random.default_rng(seed)
    return g.integers(0, 1 << 16, size=(rows, D), dtype=np.uint16)


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLD, "lru_hand.json")))
    S, n_step, bs, L = g["S"], g["n_step"], g["block_size"], g["kv_len"]
    max_ctx = 32
    hbt = np.arange(max_ctx // bs)[None, :]
    pool = _pool(max_ctx)
    buf = O.HotBuffer(1, S, n_step, max_ctx, bs, hbt, pool)
    for call in g["calls"]:
        need = call["need"]
        out, valid, st, stats = buf.swap_in([0], [L + 1], [L], np.array([need]))
        e = call["expect"]
        assert buf.slot_token[0] == e["slot_token"]
        assert buf.slot_ts[0] == e["slot_ts"]
        assert st == e["status"]
        assert stats["misses"] == e["misses"] and stats["hits"] == e["hits"]
        if "row_out" in e:
            assert out[0].tolist() == e["row_out"]


class NaiveLRU:
    """Independent model: a dict per request, victims chosen one at a time by
    scanning every slot for the smallest (last_use, slot) that is neither
    needed now nor already chosen."""

    def __init__(self, B, S, n_step):
        self.S, self.S_tot = S, S + n_step
        self.pos_of = [[None] * S for _ in range(B)]
        self.last = [[-1] * S for _ in range(B)]
        self.calls = 0

    def where(self, b, t):
        for s in range(self.S):
            if self.pos_of[b][s] == t:
                return s
        return None

    def swap(self, rows, L):
        """rows: list of (b, causal_len, list of positions)."""
        self.calls += 1
        need = {}
        for b, n, ts in rows:
            need.setdefault(b, [])
            for t in ts:
                if 0 <= t < min(n, L[b]) and t not in need[b]:
                    need[b].append(t)
        bad = set()
        for b in need:
            if len(need[b]) > self.S:
                bad.add(b)
                continue
            keep = set()
            for t in need[b]:
                s = self.where(b, t)
                if s is not None:
                    keep.add(s)
                    self.last[b][s] = self.calls
            chosen = set()
            for t in sorted(t for t in need[b] if self.where(b, t) is None):
                best = None
                for s in range(self.S):
                    if s in keep or s in chosen:
                        continue
                    if best is None or (self.last[b][s], s) < (self.last[b][best], best):
                        best = s
                chosen.add(best)
                self.pos_of[b][best] = t
                self.last[b][best] = self.calls
        out = []
        for b, n, ts in rows:
            row = []
            for t in ts:
                if t < 0 or t >= n:
                    row.append(-1)
                elif t >= L[b]:
                    row.append(b * self.S_tot + self.S + t - L[b])
                elif b in bad:
                    row.append(-1)
                else:
                    row.append(b * self.S_tot + self.where(b, t))
            out.append(row)
        return out, bad


@pytest.mark.parametrize("seed", range(12))
def test_against_naive_model_random_sequences(seed):
    g = np.random.default_rng(100 + seed)
    B, S, n_step, bs = 3, int(g.integers(2, 9)), 2, 4
    max_ctx = 40
    L = [int(x) for x in g.integers(1, 30, size=B)]
    nblk = max_ctx // bs
    hbt = g.permutation(B * nblk).reshape(B, nblk)
    pool = _pool(B * nblk * bs, seed)
    buf = O.HotBuffer(B, S, n_step, max_ctx, bs, hbt, pool)
    ref = NaiveLRU(B, S, n_step)
    for call in range(10):
        R = int(g.integers(1, 5))
        reqs = [int(x) for x in g.integers(0, B, size=R)]
        K = int(g.integers(1, 7))
        rows, clen = [], []
        for b in reqs:
            n = L[b] + int(g.integers(1, n_step + 1))
            clen.append(n)
            rows.append([int(x) for x in g.integers(-2, n + 2, size=K)])
        out, valid, st, stats = buf.swap_in(reqs, clen, L, np.array(rows))
        exp_out, bad = ref.swap(list(zip(reqs, clen, rows)), L)
        assert out.tolist() == exp_out
        assert valid.tolist() == [sum(1 for x in r if x >= 0) for r in exp_out]
        assert bool(st & O.STATUS_CAPACITY) == bool(bad)
        for b in range(B):
            assert buf.slot_token[b] == [(-1 if p is None else p) for p in ref.pos_of[b]]
            assert buf.slot_ts[b] == ref.last[b]
        _check_invariants(buf, B, L, reqs, rows, clen, bad)


def _check_invariants(buf, B, L, reqs, rows, clen, bad):
    for b in range(B):
        held = [t for t in buf.slot_token[b] if t >= 0]
        # (1) slots and positions map 1:1
        assert len(held) == len(set(held)) == len(buf.token_slot[b])
        for t, s in buf.token_slot[b].items():
            assert buf.slot_token[b][s] == t
            # (3) every hot row equals its host row
            assert np.array_equal(buf.hot[buf.hot_row(b, s)],
                                  buf.host_pool[O.host_row(buf.hbt, b, t, buf.block_size)])
    # (2) every requested committed position is resident after the call
    for b, n, ts in zip(reqs, clen, rows):
        if b in bad:
            continue
        for t in ts:
            if 0 <= t < min(n, L[b]):
                assert t in buf.token_slot[b]


def test_lru_order_invariant_no_evicted_newer_than_kept():
    # (4): after a call, no slot that was evicted had a larger ts than an
    # unneeded slot that was kept.
    g = np.random.default_rng(5)
    S, bs, max_ctx = 6, 4, 64
    hbt = np.arange(max_ctx // bs)[None, :]
    buf = O.HotBuffer(1, S, 1, max_ctx, bs, hbt, _pool(max_ctx))
    L = [60]
    for call in range(30):
        need = sorted(set(int(x) for x in g.integers(0, 60, size=int(g.integers(1, S + 1)))))
        before_tok = list(buf.slot_token[0])
        before_ts = list(buf.slot_ts[0])
        buf.swap_in([0], [61], L, np.array([need]))
        evicted = [s for s in range(S) if before_tok[s] >= 0 and buf.slot_token[0][s] != before_tok[s]]
        kept_unneeded = [s for s in range(S) if buf.slot_token[0][s] == before_tok[s]
                         and before_tok[s] not in need]
        for e in evicted:
            for k in kept_unneeded:
                assert (before_ts[e], e) < (before_ts[k], k)


def test_duplicates_and_padding_count_once():
    buf = O.HotBuffer(1, 4, 1, 16, 4, np.arange(4)[None, :], _pool(16))
    out, valid, st, stats = buf.swap_in([0, 0], [9, 9], [8], np.array([[3, 3, -1, 1], [1, 3, -5, 3]]))
    assert stats["misses"] == 2 and st == 0
    assert out[0].tolist() == [1, 1, -1, 0] and out[1].tolist() == [0, 1, -1, 1]
    assert valid.tolist() == [3, 3]


def test_topk_longer_than_context_pads():
    buf = O.HotBuffer(1, 8, 1, 16, 4, np.arange(4)[None, :], _pool(16))
    # context of 3 committed positions; row causal length 4 (one step slot)
    out, valid, st, _ = buf.swap_in([0], [4], [3], np.array([[2, 0, 1, 3, -1, -1]]))
    assert st == 0
    # misses 0, 1, 2 (ascending) fill empty slots 0, 1, 2; 3 is step slot 0 -> row 8
    assert out.tolist() == [[2, 0, 1, 8, -1, -1]]
    assert valid.tolist() == [4]


def test_reset_request_empties_slots():
    buf = O.HotBuffer(2, 2, 1, 16, 4, np.arange(8).reshape(2, 4), _pool(32))
    buf.swap_in([0, 1], [9, 9], [8, 8], np.array([[1, 2], [3, 4]]))
    buf.reset_request(0)
    assert buf.slot_token[0] == [-1, -1] and buf.slot_ts[0] == [-1, -1]
    assert buf.token_slot[0] == {} and len(buf.token_slot[1]) == 2


def test_commit_uses_victim_order_without_protection():
    # S = 3: slots hold (pos, ts) = (4, 1), (6, 2), empty. Committing two rows
    # takes the empty slot first, then the oldest (slot 0).
    bs, max_ctx = 4, 16
    pool = _pool(max_ctx)
    buf = O.HotBuffer(1, 3, 2, max_ctx, bs, np.arange(4)[None, :], pool)
    buf.swap_in([0], [9], [8], np.array([[4]]))
    buf.swap_in([0], [9], [8], np.array([[6]]))
    rows = _pool(2, seed=9)
    buf.now += 1
    assert buf.commit(0, 8, rows, buf.now)
    assert buf.slot_token[0] == [9, 6, 8]
    assert buf.slot_ts[0] == [3, 2, 3]
    assert np.array_equal(buf.host_pool[8], rows[0]) and np.array_equal(buf.host_pool[9], rows[1])
    assert np.array_equal(buf.hot[2], rows[0]) and np.array_equal(buf.hot[0], rows[1])
