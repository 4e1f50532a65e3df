"""Failure detection on the GPU without a fault: a bounded device wait that
nothing completes gives up, reports HS_STATUS_TIMEOUT in the caller's status
word, and the context keeps running kernels (an attention call afterwards
matches the oracle)."""
import time

import numpy as np
import pytest
import torch

from oracle import hs_oracle as O
from gpu_util import check_attn, lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    hs = lib()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    hs.hs_wait_probe(st, 1 << 21)          # about 1 ms of SM cycles
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert int(st.item()) == hs.HS_STATUS_TIMEOUT
    # the same context, right after: an attention call, checked as usual
    g = np.random.default_rng(5)
    q = _bf16(g.standard_normal((3, 128, 576)) / 24)
    kv = _bf16(g.standard_normal((300, 576)) / 24)
    idx = g.integers(0, 300, size=(3, 100)).astype(np.int32)
    out = torch.empty((3, 128, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((3, 128), dtype=torch.float32, device=DEV)
    st2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    hs.hs_sparse_attn_decode(q.to(DEV), kv.to(DEV), torch.as_tensor(idx, device=DEV), 0.04, out,
                             lse, st2)
    e_out, e_lse = O.sparse_attn_decode(q, kv, idx, 0.04)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    check_attn(out, e_out, lse, e_lse)
