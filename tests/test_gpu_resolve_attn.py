"""GPU parity: a1 (fully-resident index conversion) bit-exact, a6 (sparse
attention) within max abs 1e-2 and per-vector relative 2e-2 of the float64
oracle, on small ragged cases, special cases and workload 2 at full size."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import hs_oracle as O
from gpu_util import check_attn, lib, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("K", [1, 5, 64, 130, 2048])
def test_resolve_small_and_ragged(K):
    hs = lib()
    g = np.random.default_rng(K)
    B, bs, nblk, R = 5, 16, 12, 9
    bt = g.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    bt[2, 7] = -1                              # an unallocated block
    req = g.integers(0, B, size=R).astype(np.int32)
    clen = g.integers(1, nblk * bs + 1, size=R).astype(np.int32)
    topk = g.integers(-3, nblk * bs, size=(R, K)).astype(np.int32)
    for stride in (bs, 3 * bs):
        e_idx, e_valid, e_st = O.resolve_topk(req, clen, bt, topk, bs, stride)
        out = torch.full((R, K), 7, dtype=torch.int32, device=DEV)
        valid = torch.full((R,), 7, dtype=torch.int32, device=DEV)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        t = lambda a: torch.as_tensor(a, device=DEV)
        hs.hs_resolve_topk(t(req), t(clen), t(bt), t(topk), bs, stride, out, valid, st)
        torch.cuda.synchronize()
        assert np.array_equal(np_(out), e_idx)
        assert np.array_equal(np_(valid), e_valid)
        assert int(st.item()) == e_st


def _attn_case(seed, R, H, K, N, sharp=False):
    g = np.random.default_rng(seed)
    s = 1.0 if sharp else 1.0 / 24
    q = _bf16(g.standard_normal((R, H, 576)) * s)
    kv = _bf16(g.standard_normal((N, 576)) * s)
    idx = g.integers(0, N, size=(R, K)).astype(np.int32)
    if K > 3:
        idx[0, 1] = -1
        idx[0, 2] = N + 5                       # out of range: skipped
        idx[min(1, R - 1), 0] = idx[min(1, R - 1), K - 1]   # a duplicate entry
    idx[R - 1, :] = -1                          # an empty row
    return q, kv, idx


@pytest.mark.parametrize("H,K", [(16, 1), (16, 64), (64, 37), (128, 200), (80, 130),
                                 (128, 2048), (1, 65)])
@pytest.mark.parametrize("sharp", [False, True])
def test_attention_small(H, K, sharp):
    hs = lib()
    R, N = 4, 3000
    q, kv, idx = _attn_case(H * 1000 + K, R, H, K, N, sharp)
    scale = 1.0 / 24
    ref, ref_lse = O.sparse_attn_decode(q, kv, idx, scale)
    out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((R, H), dtype=torch.float32, device=DEV)
    hs.hs_sparse_attn_decode(q.to(DEV), kv.to(DEV), torch.as_tensor(idx, device=DEV), scale,
                             out, lse)
    torch.cuda.synchronize()
    check_attn(out, ref, lse, ref_lse)


@pytest.mark.parametrize("H,K", [(200, 96), (256, 130), (1024, 64)])
def test_attention_several_head_groups(H, K):
    """More than 128 heads: one CTA pair per group of 128 heads, the last
    group ragged (rows past H are zero-filled by the Q copy and not written)."""
    hs = lib()
    R, N = 3, 2000
    q, kv, idx = _attn_case(H + K, R, H, K, N)
    scale = 1.0 / 24
    ref, ref_lse = O.sparse_attn_decode(q, kv, idx, scale)
    out = torch.full((R, H, 512), 7.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((R, H), dtype=torch.float32, device=DEV)
    hs.hs_sparse_attn_decode(q.to(DEV), kv.to(DEV), torch.as_tensor(idx, device=DEV), scale,
                             out, lse)
    torch.cuda.synchronize()
    check_attn(out, ref, lse, ref_lse)


@pytest.mark.parametrize("K,sharp", [(4096, False), (8192, True)])
def test_attention_long_rows(K, sharp):
    """Rows of 128 and 256 tiles (the ring slots wrap many times; padding,
    out-of-range and duplicate entries as in the small cases)."""
    hs = lib()
    R, H, N = 2, 128, 20000
    q, kv, idx = _attn_case(K + 7, R, H, K, N, sharp)
    scale = 1.0 / 24
    ref, ref_lse = O.sparse_attn_decode(q, kv, idx, scale)
    out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((R, H), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hs.hs_sparse_attn_decode(q.to(DEV), kv.to(DEV), torch.as_tensor(idx, device=DEV), scale,
                             out, lse, st)
    torch.cuda.synchronize()
    check_attn(out, ref, lse, ref_lse)
    assert int(st.item()) == 0


def test_attention_single_valid_key_is_exact():
    hs = lib()
    g = np.random.default_rng(3)
    q = _bf16(g.standard_normal((2, 128, 576)))
    kv = _bf16(g.standard_normal((50, 576)))
    idx = np.full((2, 96), -1, np.int32)
    idx[0, 40] = 17
    idx[1, 95] = 3
    out = torch.empty((2, 128, 512), dtype=torch.bfloat16, device=DEV)
    hs.hs_sparse_attn_decode(q.to(DEV), kv.to(DEV), torch.as_tensor(idx, device=DEV), 0.1, out)
    torch.cuda.synchronize()
    assert torch.equal(out[0].cpu(), kv[17, :512].expand(128, 512))
    assert torch.equal(out[1].cpu(), kv[3, :512].expand(128, 512))


@pytest.mark.parametrize("pos", [17, 250])
def test_attention_planted_dominant_key(pos):
    # at 17 the key is in the first tile; at 250 it is far above every score
    # seen before it, so the kernel must switch to its exact-maximum pass
    hs = lib()
    g = np.random.default_rng(4)
    H, K, N = 128, 300, 400
    q = g.standard_normal((1, H, 576)) / 24
    kv = g.standard_normal((N, 576)) / 24
    q[0, :, 0] = 1.0
    kv[:, 0] = 0.0
    kv[123, 0] = 60.0                           # logit >= 50 above all others (scale 1)
    idx = g.permutation(N)[:K].astype(np.int32)
    idx[idx == 123] = idx[pos]
    idx[pos] = 123
    q, kv = _bf16(q), _bf16(kv)
    out = torch.empty((1, H, 512), dtype=torch.bfloat16, device=DEV)
    hs.hs_sparse_attn_decode(q.to(DEV), kv.to(DEV), torch.as_tensor(idx[None], device=DEV),
                             1.0, out)
    torch.cuda.synchronize()
    got = out[0].float().cpu()
    want = kv[123, :512].float().expand(H, 512)
    ulp = torch.abs(want) * 2.0 ** -7 + 1e-30
    assert ((got - want).abs() <= ulp).all()


@pytest.mark.parametrize("lead", [64, 96])
def test_attention_leading_padding(lead):
    # rows whose first `lead` entries are padding: no score to take the softmax
    # reference from until later tiles
    hs = lib()
    R, H, K, N = 3, 128, 300, 1000
    q, kv, idx = _attn_case(lead, R, H, K, N, sharp=True)
    idx[:, :lead] = -1
    scale = 1.0 / 24
    ref, ref_lse = O.sparse_attn_decode(q, kv, idx, scale)
    out = torch.empty((R, H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((R, H), dtype=torch.float32, device=DEV)
    hs.hs_sparse_attn_decode(q.to(DEV), kv.to(DEV), torch.as_tensor(idx, device=DEV), scale,
                             out, lse)
    torch.cuda.synchronize()
    check_attn(out, ref, lse, ref_lse)


def test_resolve_rows_without_a_request():
    """A row whose request id is negative gets -1 everywhere, no valid entry
    and the index status bit; the other rows of the call are unaffected."""
    hs = lib()
    g = np.random.default_rng(21)
    B, bs, nblk, R, K = 3, 16, 8, 6, 64
    bt = g.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    req = np.array([0, -1, 2, 1, -5, 0], np.int32)
    clen = np.full(R, nblk * bs, np.int32)
    topk = g.integers(-1, nblk * bs, size=(R, K)).astype(np.int32)
    t = lambda a: torch.as_tensor(a, device=DEV)
    out = torch.full((R, K), 7, dtype=torch.int32, device=DEV)
    valid = torch.full((R,), 7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hs.hs_resolve_topk(t(req), t(clen), t(bt), t(topk), bs, bs, out, valid, st)
    torch.cuda.synchronize()
    ok = req >= 0
    e_idx, e_valid, e_st = O.resolve_topk(req[ok], clen[ok], bt, topk[ok], bs, bs)
    assert e_st == 0
    assert np.array_equal(np_(out)[ok], e_idx) and np.array_equal(np_(valid)[ok], e_valid)
    assert (np_(out)[~ok] == -1).all() and (np_(valid)[~ok] == 0).all()
    assert int(st.item()) == O.STATUS_INDEX


def test_workload2_full_size():
    hs = lib()
    cfg = W.get_config(2)
    rc = W.resident_case(cfg, 0, device=DEV)
    idx = torch.empty_like(rc["topk"])
    valid = torch.empty_like(rc["req"])
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    hs.hs_resolve_topk(rc["req"], rc["clen"], rc["bt"], rc["topk"], cfg.block_size,
                       cfg.block_size, idx, valid, st)
    out = torch.empty((cfg.R, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((cfg.R, cfg.H), dtype=torch.float32, device=DEV)
    hs.hs_sparse_attn_decode(rc["q"], rc["kv"], idx, cfg.scale, out, lse)
    torch.cuda.synchronize()
    e_idx, e_valid, e_st = O.resolve_topk(rc["req_np"], rc["clen_np"], rc["bt_np"],
                                          rc["topk_np"], cfg.block_size, cfg.block_size)
    assert np.array_equal(np_(idx), e_idx) and np.array_equal(np_(valid), e_valid)
    assert int(st.item()) == e_st == 0
    # every row of the workload against the oracle (about a second of float64)
    rows = list(range(cfg.R))
    kvc = rc["kv"]
    outs, lses = O.sparse_attn_decode_rows(
        rc["q"].cpu(), lambda r: kvc[torch.as_tensor(r, device=DEV)].cpu().double().numpy(),
        e_idx, cfg.scale, rows)
    check_attn(out, np.stack([outs[r] for r in rows]), lse, np.stack([lses[r] for r in rows]),
               rows=rows)


def test_resolve_then_attention_back_to_back_sees_fresh_indices():
    """The attention is a programmatic dependent launch of the resolve before
    it: over several steps, each with new top-k positions written on the
    device and no host synchronisation between resolve and attention, every
    attention must use its own step's indices (a stale read would match an
    earlier step, not this one)."""
    hs = lib()
    g = np.random.default_rng(11)
    B, L, bs, H, K = 4, 900, 64, 128, 300
    R = B
    nblk = (L + bs) // bs + 1
    bt = g.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    kv = (torch.randn((B * nblk * bs, 576), generator=torch.Generator().manual_seed(3)) / 4).to(
        torch.bfloat16).to(DEV)
    q = (torch.randn((R, H, 576), generator=torch.Generator().manual_seed(4)) / 4).to(
        torch.bfloat16).to(DEV)
    req = np.arange(B, dtype=np.int32)
    clen = np.full(B, L, np.int32)
    d_req, d_clen, d_bt = (torch.as_tensor(x, device=DEV) for x in (req, clen, bt))
    steps = 6
    topks = [np.stack([g.permutation(L)[:K] for _ in range(R)]).astype(np.int32)
             for _ in range(steps)]
    d_topk = torch.empty((R, K), dtype=torch.int32, device=DEV)
    idx = torch.empty_like(d_topk)
    outs = [torch.empty((R, H, 512), dtype=torch.bfloat16, device=DEV) for _ in range(steps)]
    host_topk = [torch.as_tensor(t).pin_memory() for t in topks]
    for s in range(steps):
        d_topk.copy_(host_topk[s], non_blocking=True)
        hs.hs_resolve_topk(d_req, d_clen, d_bt, d_topk, bs, bs, idx)
        hs.hs_sparse_attn_decode(q, kv, idx, 0.05, outs[s])
    torch.cuda.synchronize()
    kv_np = kv.cpu()
    for s in range(steps):
        e_idx, _, _ = O.resolve_topk(req, clen, bt, topks[s], bs, bs)
        ref, _ = O.sparse_attn_decode(q.cpu(), kv_np, e_idx, 0.05)
        check_attn(outs[s], ref)


def test_chunked_rows_on_two_streams_match_one_call():
    """The rows of workload 2 in unequal chunks (43 / 42 / 29 / 14), each
    resolved and attended on one of two streams with no host synchronisation,
    give the one-call output bit for bit (rows are independent and the kernel
    is deterministic); sampled rows are checked against the oracle."""
    hs = lib()
    cfg = W.get_config(2)
    rc = W.resident_case(cfg, 0, device=DEV)
    idx_all = torch.empty_like(rc["topk"])
    out_all = torch.empty((cfg.R, cfg.H, 512), dtype=torch.bfloat16, device=DEV)
    lse_all = torch.empty((cfg.R, cfg.H), dtype=torch.float32, device=DEV)
    hs.hs_resolve_topk(rc["req"], rc["clen"], rc["bt"], rc["topk"], cfg.block_size,
                       cfg.block_size, idx_all)
    hs.hs_sparse_attn_decode(rc["q"], rc["kv"], idx_all, cfg.scale, out_all, lse_all)
    idx = torch.empty_like(rc["topk"])
    out = torch.full_like(out_all, 7.0)
    lse = torch.zeros_like(lse_all)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    start = torch.cuda.Event()
    start.record()
    cuts = [0, 43, 85, 114, cfg.R]
    for k in range(len(cuts) - 1):
        r0, r1 = cuts[k], cuts[k + 1]
        s = streams[k % 2]
        s.wait_event(start)
        hs.hs_resolve_topk(rc["req"][r0:r1], rc["clen"][r0:r1], rc["bt"], rc["topk"][r0:r1],
                           cfg.block_size, cfg.block_size, idx[r0:r1], stream=s)
        hs.hs_sparse_attn_decode(rc["q"][r0:r1], rc["kv"], idx[r0:r1], cfg.scale, out[r0:r1],
                                 lse[r0:r1], stream=s)
    torch.cuda.synchronize()
    assert torch.equal(idx, idx_all)
    assert torch.equal(out.view(torch.int16), out_all.view(torch.int16))
    assert torch.equal(lse, lse_all)
    e_idx, _, _ = O.resolve_topk(rc["req_np"], rc["clen_np"], rc["bt_np"], rc["topk_np"],
                                 cfg.block_size, cfg.block_size)
    rows = [42, 43, 84, 85, 113, 114, 127]
    kvc = rc["kv"]
    outs, lses = O.sparse_attn_decode_rows(
        rc["q"].cpu(), lambda r: kvc[torch.as_tensor(r, device=DEV)].cpu().double().numpy(),
        e_idx, cfg.scale, rows)
    check_attn(out, np.stack([outs[r] for r in rows]), lse, np.stack([lses[r] for r in rows]),
               rows=rows)
