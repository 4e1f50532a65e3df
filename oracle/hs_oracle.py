"""Plain CPU oracle for the HiSparse top-k sparse decode hot path.

TEST INFRASTRUCTURE ONLY. This module is imported by ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py``, and by nothing else. The product path (the CUDA library
and its Python binding) never imports, calls or links it, and shares no code
with it: no kernels, helpers, tables or constants. Only the seeded input
generators (``workloads.py``) feed both sides.

Everything here is the plain definition, written step by step:

* integer work (index conversion, the hot-buffer LRU, greedy verify) is a
  serial simulation in pure Python over small integers;
* attention is computed in float64 from the exact float64 value of every bf16
  input, with a library matmul as the only primitive.

Sources (pages of the hisparse_top_sparse material; the parenthesis names the
section of the page):

* "hiSparse-MTP" (Notion), section 1 (startup) and the list of core state maps:
  per-request device buffer of slots, slot -> token position, logical position
  -> slot, position -> host KV location, and "LRU slots".
* "投机解码的 KV 流转：prefill 阶段 DFlash 也要吃下整个 prompt" (shenshijiu.com),
  sections ③-⑥ and the closing table: greedy verify of [anchor, drafts], the
  correction / bonus token, which positions keep target KV, and where the next
  round's anchor and drafts sit.
* "vllm 分析(十二) HiSparse 下篇" (devpress.csdn.net), sections
  ``HiSparseCacheHandle.resolve_topk`` (fully-resident index conversion versus
  swap-in) and "数据 back up" (paged host row = block * block_size + offset).

Readings where the pages are silent:

R1  Row ``i`` of request ``b`` is the query at position ``L_b + i``; its causal
    length is ``L_b + i + 1``. ``L_b`` is the committed KV length.
R2  A hot buffer holds, per request, ``S`` LRU slots followed by ``n_step``
    step slots. Step slot ``k`` holds the freshly computed KV of position
    ``L_b + k`` (written by the caller), is always a hit and is outside the
    LRU. A position ``t`` with ``t < 0`` is padding (-1 out); ``t >=`` the
    row's causal length is an index error (-1 out, status bit 1).
R3  LRU: a per-buffer counter ``now`` goes up by one per swap-in call and per
    commit call. Hits get ``ts := now``. Victims are the slots that do not hold
    a position needed in this call, ordered by ``(ts, slot)`` ascending, empty
    slots having ``ts = -1``. The distinct missing positions of a request, in
    ascending order, go to the victims in that order and get ``ts := now``. If
    a request needs more than ``S`` distinct committed positions in one call,
    it gets status bit 2, all its committed entries come out as -1 and its
    state is left unchanged. A commit uses the same victim order with no
    protected slot.
R4  ``valid[r]`` counts the non-negative entries of row ``r``; entries keep
    their place (no compaction).
R5  Attention: entries outside ``[0, N)`` are skipped, duplicates count as
    often as they appear, a row with no valid entry gives ``out = 0`` and
    ``lse = -inf``; ``lse`` is the natural log of ``sum_j exp(scale * s_j)``.
R6  Greedy argmax ties go to the lowest vocabulary index.
R7  Host pool row of position ``t`` of request ``b`` is
    ``hbt[b][t // bs] * bs + t % bs``.
"""

from __future__ import annotations

import numpy as np
import torch

# Status bits of the device status word, as the boundary defines them.
STATUS_INDEX = 1
STATUS_CAPACITY = 2

LATENT_DIM = 576   # D: q and the latent KV row
VALUE_DIM = 512    # Dv: values are the first 512 dims of a latent row


def bf16_bits_to_f64(x) -> np.ndarray:
    """Exact float64 value of bf16 data given as a torch bf16 tensor or as
    raw uint16/int16 bit patterns."""
    if isinstance(x, torch.Tensor):
        if x.dtype == torch.bfloat16:
            return x.detach().cpu().to(torch.float64).numpy()
        x = x.detach().cpu().numpy()
    u = np.asarray(x).view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def _np_i64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.asarray(x).astype(np.int64)


def _rows_u16(x) -> np.ndarray:
    """A bf16 array as raw uint16 bit patterns (row copies stay bit-exact)."""
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            x = x.view(torch.int16)
        x = x.numpy()
    return np.asarray(x).view(np.uint16)


# --------------------------------------------------------------------------
# Host pool addressing ("vllm 分析(十二) HiSparse 下篇", 数据 back up)
# --------------------------------------------------------------------------

def host_row(hbt, b: int, t: int, block_size: int) -> int:
    """Row of the paged host pool that holds position ``t`` of request ``b``:
    the host block that covers ``t`` times the block size, plus the offset of
    ``t`` inside the block (reading R7)."""
    return int(hbt[b][t // block_size]) * block_size + t % block_size


# --------------------------------------------------------------------------
# a1: fully-resident index conversion
#     ("vllm 分析(十二) HiSparse 下篇", HiSparseCacheHandle.resolve_topk)
# --------------------------------------------------------------------------

def resolve_topk(req_id_per_row, row_causal_len, block_table, topk,
                 block_size: int, phys_block_stride: int):
    """Physical cache row of every top-k position of every query row.

    For row ``r`` of request ``b = req_id_per_row[r]`` and entry ``t``:
    ``block_table[b][t // block_size] * phys_block_stride + t % block_size``.
    Padding (``t < 0``) gives -1; ``t >= row_causal_len[r]`` or a negative
    block-table entry gives -1 and sets the index status bit.

    Returns ``(idx int32 [R][K], valid int32 [R], status int)``.
    """
    req = _np_i64(req_id_per_row)
    clen = _np_i64(row_causal_len)
    bt = _np_i64(block_table)
    tk = _np_i64(topk)
    R, K = tk.shape
    idx = np.full((R, K), -1, dtype=np.int32)
    valid = np.zeros(R, dtype=np.int32)
    status = 0
    for r in range(R):
        b = int(req[r])
        for j in range(K):
            t = int(tk[r, j])
            if t < 0:
                continue
            if t >= clen[r]:
                status |= STATUS_INDEX
                continue
            blk = int(bt[b, t // block_size])
            if blk < 0:
                status |= STATUS_INDEX
                continue
            idx[r, j] = blk * phys_block_stride + t % block_size
            valid[r] += 1
    return idx, valid, status


# --------------------------------------------------------------------------
# a2-a5, a8: the per-request device hot buffer with its LRU slots
#     ("hiSparse-MTP", section 1 and the core state maps;
#      "vllm 分析(十二) HiSparse 下篇", resolve_topk -> runtime.swap_in)
# --------------------------------------------------------------------------

class HotBuffer:
    """State of the hot buffer: for each request ``b``

    * ``slot_token[b][s]``  position held by LRU slot ``s`` (-1 = empty),
    * ``slot_ts[b][s]``     last-use stamp of slot ``s`` (-1 = empty),
    * ``token_slot[b][t]``  slot holding committed position ``t`` (-1 = none),
    * ``hot[b * S_tot + s]`` the 576 bf16 values of the row in slot ``s``
      (LRU slots ``0..S-1``, step slots ``S..S_tot-1``, reading R2),

    plus the host pool (paged, reading R7) and the call counter ``now``.
    """

    def __init__(self, max_reqs: int, S: int, n_step: int, max_ctx: int,
                 block_size: int, hbt, host_pool):
        self.max_reqs = max_reqs
        self.S = S
        self.n_step = n_step
        self.S_tot = S + n_step
        self.max_ctx = max_ctx
        self.block_size = block_size
        self.hbt = _np_i64(hbt)
        # host pool rows and hot rows are kept as raw bf16 bits
        self.host_pool = _rows_u16(host_pool)
        self.slot_token = [[-1] * S for _ in range(max_reqs)]
        self.slot_ts = [[-1] * S for _ in range(max_reqs)]
        self.token_slot = [dict() for _ in range(max_reqs)]
        self.hot = np.zeros((max_reqs * self.S_tot, LATENT_DIM), dtype=np.uint16)
        self.now = 0
        self.last_plan = []

    # -- queries ---------------------------------------------------------
    def token_slot_array(self, b: int) -> np.ndarray:
        out = np.full(self.max_ctx, -1, dtype=np.int32)
        for t, s in self.token_slot[b].items():
            out[t] = s
        return out

    def hot_row(self, b: int, s: int) -> int:
        return b * self.S_tot + s

    # -- admit -----------------------------------------------------------
    def reset_request(self, b: int) -> None:
        """Empty every slot of request ``b`` (a request admitted into the
        decode batch starts with an empty device buffer: "hiSparse-MTP",
        section 3, collect_ready_reqs)."""
        self.slot_token[b] = [-1] * self.S
        self.slot_ts[b] = [-1] * self.S
        self.token_slot[b] = {}

    # -- LRU helpers -------------------------------------------------------
    def _victim_order(self, b: int, protected: set) -> list:
        """Slots not in ``protected``, least recently used first: ascending
        ``(ts, slot)``, so empty slots (ts = -1) lead in slot order (R3)."""
        cand = [s for s in range(self.S) if s not in protected]
        return sorted(cand, key=lambda s: (self.slot_ts[b][s], s))

    def _place(self, b: int, s: int, t: int, now: int) -> None:
        old = self.slot_token[b][s]
        if old >= 0:
            del self.token_slot[b][old]
        self.slot_token[b][s] = t
        self.token_slot[b][t] = s
        self.slot_ts[b][s] = now

    # -- a2-a5: swap-in ------------------------------------------------------
    def swap_in(self, req_id_per_row, row_causal_len, kv_len, topk):
        """Make every committed position named by ``topk`` resident and return
        the hot-row index table.

        Returns ``(slot_idx int32 [R][K], valid int32 [R], status int,
        stats dict)``; ``stats`` holds ``misses`` (rows copied from the host
        pool) and ``hits``.
        """
        self.now += 1
        now = self.now
        req = _np_i64(req_id_per_row)
        clen = _np_i64(row_causal_len)
        L = _np_i64(kv_len)
        tk = _np_i64(topk)
        R, K = tk.shape
        status = 0

        # a2: the distinct committed positions each request needs in this call
        needed: dict[int, set] = {}
        for r in range(R):
            b = int(req[r])
            needed.setdefault(b, set())
            for j in range(K):
                t = int(tk[r, j])
                if t < 0:
                    continue
                if t >= clen[r]:
                    status |= STATUS_INDEX
                    continue
                if t >= L[b]:
                    continue          # step slot: always a hit, outside the LRU
                needed[b].add(t)

        failed = set()
        hits = misses = 0
        self.last_plan = []       # (request, slot, position) of every copy made
        for b in sorted(needed):
            need = needed[b]
            if len(need) > self.S:
                status |= STATUS_CAPACITY
                failed.add(b)
                continue
            resident = sorted(t for t in need if t in self.token_slot[b])
            missing = sorted(t for t in need if t not in self.token_slot[b])
            hits += len(resident)
            protected = set()
            for t in resident:
                s = self.token_slot[b][t]
                self.slot_ts[b][s] = now
                protected.add(s)
            # a3: victims in LRU order, misses ascending, paired in order
            victims = self._victim_order(b, protected)
            assert len(victims) >= len(missing)
            for t, s in zip(missing, victims):
                self._place(b, s, t, now)
                # a4: copy the host row into the hot slot
                self.hot[self.hot_row(b, s)] = self.host_pool[
                    host_row(self.hbt, b, t, self.block_size)]
                self.last_plan.append((b, s, t))
            misses += len(missing)

        # a5: slot index table
        out = np.full((R, K), -1, dtype=np.int32)
        valid = np.zeros(R, dtype=np.int32)
        for r in range(R):
            b = int(req[r])
            for j in range(K):
                t = int(tk[r, j])
                if t < 0 or t >= clen[r]:
                    continue
                if t >= L[b]:
                    out[r, j] = self.hot_row(b, self.S + (t - int(L[b])))
                elif b in failed:
                    continue
                else:
                    out[r, j] = self.hot_row(b, self.token_slot[b][t])
                valid[r] += 1
        return out, valid, status, {"hits": hits, "misses": misses}

    # -- a8: commit of the accepted prefix ---------------------------------
    def commit(self, b: int, L: int, rows_u16: np.ndarray, now: int) -> bool:
        """Commit KV rows for positions ``L .. L + n - 1`` of request ``b``:
        host pool rows and LRU hot slots (victims with no protected slot).
        Returns False (state untouched) if the positions do not fit."""
        n = rows_u16.shape[0]
        if L + n > self.max_ctx or n > self.S:
            return False
        for k in range(n):
            self.host_pool[host_row(self.hbt, b, L + k, self.block_size)] = rows_u16[k]
        victims = self._victim_order(b, set())
        for k in range(n):
            s = victims[k]
            self._place(b, s, L + k, now)
            self.hot[self.hot_row(b, s)] = rows_u16[k]
        return True


# --------------------------------------------------------------------------
# a6: sparse attention over the selected latent rows
#     (DSA attention over the rows resolve_topk / swap_in return; shapes of
#      the MLA latent: 576-dim rows, values = first 512 dims)
# --------------------------------------------------------------------------

def sparse_attn_decode(q, kv, idx, scale: float):
    """For each query row ``r`` and head ``h``::

        s_j      = scale * <q[r, h, :], kv[idx[r, j], :]>          (576 dims)
        p_j      = exp(s_j) / sum_j' exp(s_j')                     (valid j)
        out[r,h] = sum_j p_j * kv[idx[r, j], 0:512]
        lse[r,h] = log(sum_j exp(s_j))

    in float64 (reading R5 for padding, duplicates and empty rows).
    ``q`` [R][H][576] and ``kv`` [N][576] are bf16 (tensor or raw bits),
    ``idx`` is int [R][K]. Returns float64 ``out`` [R][H][512], ``lse`` [R][H].
    """
    qf = bf16_bits_to_f64(q)
    kvf = kv if (isinstance(kv, np.ndarray) and kv.dtype == np.float64) else bf16_bits_to_f64(kv)
    ix = _np_i64(idx)
    R, H, D = qf.shape
    assert D == LATENT_DIM and kvf.shape[1] == LATENT_DIM
    N = kvf.shape[0]
    out = np.zeros((R, H, VALUE_DIM), dtype=np.float64)
    lse = np.full((R, H), -np.inf, dtype=np.float64)
    for r in range(R):
        rows = [int(j) for j in ix[r] if 0 <= j < N]
        if not rows:
            continue
        Kr = kvf[rows]                      # [n][576], duplicates kept
        s = scale * (qf[r] @ Kr.T)          # [H][n]
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1)
        out[r] = (p @ Kr[:, :VALUE_DIM]) / l[:, None]
        lse[r] = m[:, 0] + np.log(l)
    return out, lse


def sparse_attn_decode_rows(q, kv_rows_of, idx, scale: float, rows):
    """The same definition for a chosen subset of query rows, fetching KV rows
    through ``kv_rows_of(list_of_indices) -> float64 [n][576]`` so that a
    large cache never has to be converted whole. Returns dicts keyed by row."""
    qf_all = q
    ix = _np_i64(idx)
    outs, lses = {}, {}
    for r in rows:
        qf = bf16_bits_to_f64(qf_all[r])
        H = qf.shape[0]
        sel = [int(j) for j in ix[r] if j >= 0]
        o = np.zeros((H, VALUE_DIM))
        ls = np.full(H, -np.inf)
        if sel:
            Kr = kv_rows_of(sel)
            s = scale * (qf @ Kr.T)
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            l = p.sum(axis=1)
            o = (p @ Kr[:, :VALUE_DIM]) / l[:, None]
            ls = m[:, 0] + np.log(l)
        outs[r] = o
        lses[r] = ls
    return outs, lses


# --------------------------------------------------------------------------
# next-3: reclaim of resident pages and a batch mixing both kinds of request
#     ("vllm 分析(十二) HiSparse 下篇": reclaim_resident_blocks with
#      reclaimable_pages / release_resident_page, and the fully_resident flag
#      that HiSparseCacheHandle.resolve_topk branches on)
# --------------------------------------------------------------------------

def reclaimable_pages(block_table, n_blocks) -> list:
    """``(request, logical block)`` of every page a reclaim may release: the
    pages each request still holds (entry >= 0) except its last two logical
    blocks, listed request by request, blocks ascending (reading R16)."""
    bt = _np_i64(block_table)
    nb = _np_i64(n_blocks)
    out = []
    for b in range(bt.shape[0]):
        n = min(max(int(nb[b]), 0), bt.shape[1])
        for i in range(n - 2):
            if bt[b, i] >= 0:
                out.append((b, i))
    return out


def reclaim_resident(block_table, n_blocks, need: int):
    """Release the first ``need`` reclaimable pages: each one's entry becomes
    -1 (release_resident_page) and its block id is handed back. A request that
    lost a page is no longer fully resident.

    Returns ``(table int32 [B][stride], freed int32 [need] (-1 past the last
    release), fully_resident int32 [B], n_freed)``."""
    bt = _np_i64(block_table).copy()
    nb = _np_i64(n_blocks)
    freed = np.full(need, -1, dtype=np.int32)
    take = reclaimable_pages(bt, nb)[:need]
    for k, (b, i) in enumerate(take):
        freed[k] = bt[b, i]
        bt[b, i] = -1
    fully = np.zeros(bt.shape[0], dtype=np.int32)
    for b in range(bt.shape[0]):
        n = min(max(int(nb[b]), 0), bt.shape[1])
        fully[b] = int(all(bt[b, i] >= 0 for i in range(n)))
    return bt.astype(np.int32), freed, fully, len(take)


def sparse_attn_decode_mixed(q, kv_resident, kv_hot, row_req, fully_resident, idx,
                             scale: float):
    """``sparse_attn_decode`` for a batch mixing both kinds of request: row
    ``r`` reads ``kv_resident`` while its request is fully resident
    (``fully_resident[row_req[r]] != 0``) and ``kv_hot`` otherwise, each
    row's entries valid within its own cache (reading R17). A request id
    outside the flags leaves the row with no valid entry. ``row_req`` None
    indexes the flags by row; ``fully_resident`` None sends every row to
    ``kv_resident``."""
    qb = _rows_u16(q) if not isinstance(q, np.ndarray) else q
    as_f64 = lambda kv: kv if (isinstance(kv, np.ndarray) and kv.dtype == np.float64) \
        else bf16_bits_to_f64(kv)
    kv_resident = as_f64(kv_resident)
    kv_hot = as_f64(kv_hot) if fully_resident is not None else None
    ix = _np_i64(idx)
    R = ix.shape[0]
    H = qb.shape[1]
    out = np.zeros((R, H, VALUE_DIM), dtype=np.float64)
    lse = np.full((R, H), -np.inf, dtype=np.float64)
    for r in range(R):
        if fully_resident is None:
            kv = kv_resident
        else:
            fr = _np_i64(fully_resident)
            b = int(_np_i64(row_req)[r]) if row_req is not None else r
            if not 0 <= b < fr.shape[0]:
                continue
            kv = kv_resident if fr[b] != 0 else kv_hot
        o, l = sparse_attn_decode(qb[r:r + 1], kv, ix[r:r + 1], scale)
        out[r], lse[r] = o[0], l[0]
    return out, lse


# --------------------------------------------------------------------------
# a7-a8: greedy verify and commit of the accepted prefix
#     ("投机解码的 KV 流转", sections ④-⑥ and the closing table)
# --------------------------------------------------------------------------

def argmax_lowest(row) -> int:
    """Index of the largest logit, the lowest index among equals (R6)."""
    v = np.asarray(row)
    assert np.all(np.isfinite(v)), "logits must be finite"
    # numpy documents that argmax returns the first occurrence of the maximum
    return int(np.argmax(v))


def greedy_accept(preds, drafts):
    """Target input ``i`` (the anchor for ``i = 0``, draft ``i`` otherwise)
    yields ``preds[i]``, which checks draft ``i`` (0-based ``drafts[i]`` is
    the ``i+1``-th candidate). ``m`` is the length of the longest agreeing
    prefix; the next token is ``preds[m]``: the correction at the first
    mismatch, or the bonus token after all ``d`` drafts pass.
    Returns ``(m, next_token)``."""
    d = len(drafts)
    m = 0
    while m < d and int(drafts[m]) == int(preds[m]):
        m += 1
    return m, int(preds[m])


def verify_finalize(buf: HotBuffer, logits, drafts, step_kv, kv_len):
    """Greedy verify of every request, then commit of the accepted prefix.

    ``logits`` [B][d+1][V] (float32 or bf16), ``drafts`` int [B][d],
    ``step_kv`` bf16 [B][d+1][576] (target KV of inputs anchor, draft 1..d),
    ``kv_len`` int [B]. The KV of inputs ``0..m`` (positions ``L..L+m``) is
    kept: written to the host pool and placed in LRU slots; ``L`` grows by
    ``m + 1``. The token chosen last has no KV yet.

    Returns ``(accept_len [B], next_token [B], new_kv_len [B], status)``.
    """
    buf.now += 1
    now = buf.now
    if isinstance(logits, torch.Tensor):
        lg = logits.detach().cpu().to(torch.float64).numpy()
    else:
        lg = np.asarray(logits, dtype=np.float64)
    dr = _np_i64(drafts)
    kvb = _rows_u16(step_kv)
    L = _np_i64(kv_len).copy()
    B, d1, V = lg.shape
    acc = np.zeros(B, dtype=np.int32)
    nxt = np.zeros(B, dtype=np.int32)
    status = 0
    for b in range(B):
        preds = [argmax_lowest(lg[b, i]) for i in range(d1)]
        m, tok = greedy_accept(preds, dr[b, :d1 - 1])
        acc[b] = m
        nxt[b] = tok
        ok = buf.commit(b, int(L[b]), kvb[b, :m + 1], now)
        if ok:
            L[b] += m + 1
        else:
            status |= STATUS_CAPACITY
    return acc, nxt, L.astype(np.int32), status


# ---------------------------------------------------------------------------
# next-1: one swap plan applied to follower caches
# ---------------------------------------------------------------------------

def apply_plan(plan, follower_hot, follower_pool, hbt, block_size: int, S_tot: int,
               row_offset: int = 0) -> None:
    """A follower cache repeats the leader's latest swap-in ("vllm 分析(十二)
    HiSparse 下篇", ``HiSparseCacheHandle.resolve_topk``: a handle with a leader
    calls ``runtime.apply_plan`` with ``plan_row_offset`` instead of
    ``swap_in``; the leader's ``swap_in`` is asked to ``produce_plan``).

    ``plan`` is ``HotBuffer.last_plan``: the (request b, slot s, position t)
    of every row the leader copied. The follower has the same hot-buffer
    geometry and the same paged host pool, so each copy is repeated from the
    follower's pool into the follower's buffer (reading R14):
    ``follower_hot[row_offset + b * S_tot + s] = follower_pool[host_row(b, t)]``.
    The leader's slot table then indexes the follower's buffer unchanged.
    ``follower_hot`` and ``follower_pool`` are row arrays of any row format
    (bf16 bits, or the raw bytes of an FP8 / FP4 row), updated in place.
    """
    h = _np_i64(hbt)
    for (b, s, t) in plan:
        follower_hot[row_offset + b * S_tot + s] = follower_pool[host_row(h, b, t, block_size)]


# ---------------------------------------------------------------------------
# next-2: backup of device pages to the host caches
# ---------------------------------------------------------------------------

def backup_pages(src_layers, dst_layers, src_blocks, dst_blocks, page_offsets,
                 blocks_per_kv_block: int, block_rows: int) -> None:
    """Copy whole pages of several layers' device caches to their host caches
    ("vllm 分析(十二) HiSparse 下篇", section 数据 back up:
    ``HiSparseWorker._enqueue_transfers`` and ``hisparse_backup_layers``).

    For transfer ``i`` and layer ``l`` (reading R15): rows
    ``src_blocks[l][i] * block_rows + o`` of ``src_layers[l]`` go to rows
    ``(dst_blocks[i] * blocks_per_kv_block + page_offsets[i]) * block_rows + o``
    of ``dst_layers[l]``, for ``o = 0 .. block_rows - 1``: the source row uses
    the layer's own resident block, the host page is shared by the layers.
    Row arrays are numpy arrays of raw row contents, updated in place.
    """
    sb = _np_i64(src_blocks)
    db = _np_i64(dst_blocks)
    po = _np_i64(page_offsets)
    for l in range(len(src_layers)):
        for i in range(len(db)):
            host_page = int(db[i]) * blocks_per_kv_block + int(po[i])
            for o in range(block_rows):
                dst_layers[l][host_page * block_rows + o] = src_layers[l][int(sb[l][i]) * block_rows + o]


# ---------------------------------------------------------------------------
# next-4: row backup by slot mapping and the indexer cache's host slots
#     ("vllm 分析(十二) HiSparse 下篇", section c4a kv cache 写入:
#      runtime.backup_rows, compress_hisparse_slot_mapping,
#      hisparse_backup_indexer with its token_stride)
# ---------------------------------------------------------------------------

def backup_rows(src_layers, dst_layers, src_slots, dst_slots) -> int:
    """Copy the rows a step wrote to the host caches: for every entry ``i``
    whose two slots are non-negative and every layer ``l``,
    ``dst_layers[l][dst_slots[i]] = src_layers[l][src_slots[i]]``. A row is
    one token's entry of ``token_stride`` bytes (reading R19), here one row of
    a numpy array of raw bytes. A negative slot means "no entry"; a slot past
    the end of its array is skipped and reported. Returns the status bits."""
    ss = _np_i64(src_slots)
    ds = _np_i64(dst_slots)
    status = 0
    for i in range(len(ss)):
        s, d = int(ss[i]), int(ds[i])
        if s < 0 or d < 0:
            continue
        if s >= len(src_layers[0]) or d >= len(dst_layers[0]):
            status |= STATUS_INDEX
            continue
        for l in range(len(src_layers)):
            dst_layers[l][d] = src_layers[l][s]
    return status


def compress_slot_mapping(host_slots, positions, storage_block_size: int,
                          compress_ratio: int) -> np.ndarray:
    """Host row of each token in the indexer's compressed host cache (reading
    R18): a logical block of ``storage_block_size * compress_ratio`` token
    slots is stored as one block of ``storage_block_size`` entries, one entry
    per ``compress_ratio`` consecutive positions, so the token at ``position``
    with logical host slot ``slot`` lands in entry
    ``(position mod logical block size) // compress_ratio`` of storage block
    ``slot // logical block size``. Negative inputs give -1."""
    lbs = storage_block_size * compress_ratio
    out = np.full(len(host_slots), -1, dtype=np.int64)
    for i, (s, p) in enumerate(zip(_np_i64(host_slots), _np_i64(positions))):
        if s < 0 or p < 0:
            continue
        block = int(s) // lbs
        entry = (int(p) % lbs) // compress_ratio
        out[i] = block * storage_block_size + entry
    return out
