"""hs_verify_accept_noalloc: the acceptance half of hs_verify_finalize for
callers that cannot allocate device memory (its scratch is a static array
inside the library). Called through the C ABI twice in a row, it must give the
same accepted lengths and next tokens as hs_verify_finalize on the same
inputs. Collected last so that a run stopping at the first failure has run
every other test first."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import hs_oracle as O
from gpu_util import lib, np_

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _finalize_reference(hs, logits, drafts, B, d):
    """accept_len / next_token from hs_verify_finalize on a throwaway buffer."""
    S, bs = 8, 16
    max_ctx = 64
    pool = torch.zeros((B * max_ctx, 576), dtype=torch.bfloat16).pin_memory()
    hot = torch.zeros((B * (S + d + 1), 576), dtype=torch.bfloat16, device=DEV)
    hbt = torch.arange(B * (max_ctx // bs), dtype=torch.int32, device=DEV).view(B, -1)
    buf = hs.HsBuffer(B, S, d + 1, max_ctx, bs, hot, pool, hbt)
    kv_len = torch.full((B,), 5, dtype=torch.int32, device=DEV)
    skv = torch.zeros((B, d + 1, 576), dtype=torch.bfloat16, device=DEV)
    acc = torch.empty(B, dtype=torch.int32, device=DEV)
    nxt = torch.empty_like(acc)
    hs.hs_verify_finalize(buf, logits, drafts, skv, kv_len, acc, nxt)
    assert hs.hs_get_status(buf) == 0
    buf.close()
    return np_(acc), np_(nxt)


@pytest.mark.parametrize("dtype,V", [(torch.float32, 1024), (torch.bfloat16, 129280)])
def test_noalloc_accept_matches_verify_finalize_twice(dtype, V):
    hs = lib()
    B, d = 64, 3
    for call in range(2):
        cfg = W.get_config(1)
        cfg.B, cfg.V, cfg.seed = B, V, 40 + call
        cfg.logits_dtype = "f32" if dtype == torch.float32 else "bf16"
        logits, drafts, _ = W.planted_logits(cfg, device=DEV)
        t_drafts = torch.as_tensor(drafts, device=DEV)
        want_acc, want_nxt = _finalize_reference(hs, logits, t_drafts, B, d)
        acc = torch.full((B,), -7, dtype=torch.int32, device=DEV)
        nxt = torch.full((B,), -7, dtype=torch.int32, device=DEV)
        hs.hs_verify_accept_noalloc(logits, t_drafts, acc, nxt)
        torch.cuda.synchronize()
        assert np.array_equal(np_(acc), want_acc)
        assert np.array_equal(np_(nxt), want_nxt)


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    hs = lib()
    logits = torch.zeros((20000, 4, 8), dtype=torch.float32, device=DEV)  # 80000 rows
    drafts = torch.zeros((20000, 3), dtype=torch.int32, device=DEV)
    acc = torch.empty(20000, dtype=torch.int32, device=DEV)
    with pytest.raises(hs.HisparseError, match="static scratch"):
        hs.hs_verify_accept_noalloc(logits, drafts, acc, acc.clone())


def test_noalloc_at_the_static_scratch_limit():
    """B * (d + 1) = 65536 rows, the most the static scratch takes, twice (the
    per-request row counts must be back at 0 after the first call); ties
    are frequent (integer logits) and half the drafts are planted as the
    argmax; every request against the oracle's argmax and acceptance."""
    hs = lib()
    B, d, V = 16384, 3, 64
    g = np.random.default_rng(77)
    for call in range(2):
        lg = g.integers(-4, 5, size=(B, d + 1, V)).astype(np.float32)
        drafts = g.integers(0, V, size=(B, d)).astype(np.int32)
        plant = g.random((B, d)) < 0.5
        for b, i in zip(*np.nonzero(plant)):
            drafts[b, i] = int(np.argmax(lg[b, i]))
        acc = torch.full((B,), -7, dtype=torch.int32, device=DEV)
        nxt = torch.full((B,), -7, dtype=torch.int32, device=DEV)
        hs.hs_verify_accept_noalloc(torch.as_tensor(lg, device=DEV),
                                    torch.as_tensor(drafts, device=DEV), acc, nxt)
        torch.cuda.synchronize()
        want = [O.greedy_accept([O.argmax_lowest(lg[b, i]) for i in range(d + 1)], drafts[b])
                for b in range(B)]
        assert np_(acc).tolist() == [m for m, _ in want]
        assert np_(nxt).tolist() == [t for _, t in want]
