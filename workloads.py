"""Seeded synthetic inputs for the HiSparse top-k sparse decode path.

This module is shared by the CUDA path's tests/bench and by the CPU oracle. It
only draws inputs; it holds none of the method's arithmetic (no index
conversion, no LRU, no attention, no verify).

The five workloads follow the shapes of the material's workloads:

1. tiny offload decode: 2 requests with context 512 and 300, block 64,
   anchor + 3 drafts, 16 heads, top-k 64, 128 hot slots, 2 steps, greedy
   verify over 1024 fp32 logits;
2. fully resident: 32 x 8192 context, shuffled physical block table, 128
   heads, top-k 2048; resolve + attention;
3. host backed with locality: 64 x 32768 context, 4096 hot slots, top-k 2048,
   80 % of positions repeat the previous step's set, 16 steps;
4. long mixed: 128 requests with context uniform in [16384, 131072], 4096 hot
   slots, 90 % reuse, 8 steps;
5. verify + finalize: 256 x 4096 context, 3 drafts, 4 x 129280 bf16 logits,
   drafts planted as the argmax with probability 0.7.

Values: q and KV latent rows are N(0, 1) / 24 rounded to bf16; logits are
N(0, 1). Random streams are keyed by (seed, what, step, request) so any part
can be redrawn alone.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

LATENT = 576
KV_SCALE = 1.0 / 24.0


@dataclass
class Config:
    no: int
    name: str
    B: int
    L: list                  # committed KV length per request at step 0
    block_size: int = 64
    d: int = 3               # drafts per request (rows per request = d + 1)
    H: int = 128
    K: int = 2048
    S: int = 0               # LRU hot slots per request (0: fully resident)
    steps: int = 1
    reuse: float = 0.0       # share of a request's set kept from the last step
    V: int = 0               # vocabulary (verify)
    logits_dtype: str = "f32"
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def R(self) -> int:
        return self.B * (self.d + 1)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(LATENT)


def _lengths_cfg4(seed: int) -> list:
    g = rng(seed, "ctx")
    return [int(x) for x in g.integers(16384, 131072 + 1, size=128)]


def get_config(no: int) -> Config:
    if no == 1:
        return Config(1, "tiny-offload-2x(512,300)-h16-k64-s128", B=2, L=[512, 300],
                      H=16, K=64, S=128, steps=2, V=1024, logits_dtype="f32", seed=0)
    if no == 2:
        return Config(2, "fully-resident-32x8192-h128-k2048", B=32, L=[8192] * 32,
                      seed=2)
    if no == 3:
        return Config(3, "host-backed-64x32768-s4096-k2048-reuse0.8", B=64,
                      L=[32768] * 64, S=4096, steps=16, reuse=0.8, seed=3)
    if no == 4:
        return Config(4, "long-mixed-128x[16384,131072]-s4096-k2048-reuse0.9", B=128,
                      L=_lengths_cfg4(4), S=4096, steps=8, reuse=0.9, seed=4)
    if no == 5:
        return Config(5, "verify-finalize-256x4096-v129280", B=256, L=[4096] * 256,
                      S=4096, V=129280, logits_dtype="bf16", seed=5)
    raise ValueError(no)


# ---------------------------------------------------------------- streams --

_TAGS = {}


def _tag(what: str) -> int:
    if what not in _TAGS:
        _TAGS[what] = sum((i + 1) * ord(c) for i, c in enumerate(what)) & 0xFFFFFF
    return _TAGS[what]


def rng(seed: int, what: str, *keys: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(
        np.random.SeedSequence([seed, _tag(what), *[int(k) for k in keys]])))


def torch_seed(seed: int, what: str, *keys: int) -> int:
    return int(np.random.SeedSequence([seed, _tag(what), *[int(k) for k in keys]])
               .generate_state(1, dtype=np.uint64)[0] & ((1 << 63) - 1))


def bf16_normal(shape, scale: float, seed: int, what: str, *keys, device="cpu",
                chunk_rows: int = 1 << 20) -> torch.Tensor:
    """N(0, 1) * scale rounded to bf16, drawn with a seeded torch generator on
    ``device``. Large leading dimensions are drawn in chunks, each with its own
    key, so memory stays bounded."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    n0 = shape[0]
    for c, start in enumerate(range(0, n0, chunk_rows)):
        stop = min(n0, start + chunk_rows)
        g = torch.Generator(device=device)
        g.manual_seed(torch_seed(seed, what, *keys, c))
        x = torch.randn((stop - start,) + shape[1:], generator=g, device=device,
                        dtype=torch.float32)
        out[start:stop] = (x * scale).to(torch.bfloat16)
    return out


# ------------------------------------------------------------ structure --

def rows_of(cfg: Config):
    """req_id and in-request row index of every query row (requests in order,
    rows 0..d inside each request)."""
    req = np.repeat(np.arange(cfg.B, dtype=np.int32), cfg.d + 1)
    row_in_req = np.tile(np.arange(cfg.d + 1, dtype=np.int32), cfg.B)
    return req, row_in_req


def causal_lengths(L, req, row_in_req) -> np.ndarray:
    """Causal length L_b + i + 1 of each query row (row i sits at L_b + i)."""
    L = np.asarray(L, dtype=np.int64)
    return (L[req] + row_in_req + 1).astype(np.int32)


def shuffled_block_table(seed: int, what: str, blocks_per_req) -> tuple:
    """Block table whose entries are a random permutation of all physical
    blocks. ``blocks_per_req`` is a list; rows are padded with -1.
    Returns (table int32 [B][max_blocks], total_blocks)."""
    blocks_per_req = [int(n) for n in blocks_per_req]
    total = sum(blocks_per_req)
    perm = rng(seed, what).permutation(total).astype(np.int32)
    width = max(blocks_per_req)
    bt = np.full((len(blocks_per_req), width), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(blocks_per_req):
        bt[b, :n] = perm[pos:pos + n]
        pos += n
    return bt, total


def distinct_uniform(g: np.random.Generator, n_candidates: int, k: int) -> np.ndarray:
    """``min(k, n)`` distinct values uniform in [0, n), in random order, padded
    with -1 to length k."""
    take = min(k, n_candidates)
    out = np.full(k, -1, dtype=np.int32)
    if take > 0:
        out[:take] = g.choice(n_candidates, size=take, replace=False)
    return out


def topk_independent(cfg: Config, step: int, L, req, row_in_req) -> np.ndarray:
    """Each row draws K distinct positions uniform below its causal length
    (workloads 1 and 2)."""
    clen = causal_lengths(L, req, row_in_req)
    out = np.empty((len(req), cfg.K), dtype=np.int32)
    for r in range(len(req)):
        g = rng(cfg.seed, "topk", step, r)
        out[r] = distinct_uniform(g, int(clen[r]), cfg.K)
    return out


def _fresh(g, lo: int, hi: int, n: int, taken: set) -> list:
    """Up to ``n`` values uniform in [lo, hi), distinct from ``taken`` and
    from each other (``taken`` is updated)."""
    free = (hi - lo) - sum(1 for x in taken if lo <= x < hi)
    n = max(0, min(n, free))
    got = []
    while len(got) < n:
        x = int(g.integers(lo, hi))
        if x not in taken:
            taken.add(x)
            got.append(x)
    return got


def locality_sets(cfg: Config, L_b: int, b: int, steps: int) -> list:
    """Per-request position sets of workloads 3 and 4: step 0 is K distinct
    positions uniform in [0, L); step t keeps a uniform ``reuse`` share of the
    previous set and draws the rest fresh (not in the previous set) and
    distinct, half from the last 4096 positions and half uniform in [0, L)."""
    K = cfg.K
    sets = []
    g = rng(cfg.seed, "set", b)
    cur = [int(x) for x in g.choice(L_b, size=min(K, L_b), replace=False)]
    sets.append(np.array(cur, dtype=np.int32))
    n_keep = int(round(cfg.reuse * K))
    for t in range(1, steps):
        g = rng(cfg.seed, "set", b, t)
        keep = [cur[i] for i in g.choice(len(cur), size=min(n_keep, len(cur)), replace=False)]
        taken = set(cur)          # fresh positions are new to the request
        n_new = K - len(keep)
        recent = _fresh(g, max(0, L_b - 4096), L_b, n_new // 2, taken)
        anywhere = _fresh(g, 0, L_b, n_new - len(recent), taken)
        cur = keep + recent + anywhere
        sets.append(np.array(cur, dtype=np.int32))
    return sets


def topk_shared_sets(cfg: Config, sets_per_req: list, step: int) -> np.ndarray:
    """Rows of a request share the step's set, each row in its own shuffled
    order (workloads 3, 4 and the warm-up of 5)."""
    rows = cfg.d + 1
    out = np.full((cfg.B * rows, cfg.K), -1, dtype=np.int32)
    for b in range(cfg.B):
        s = sets_per_req[b][step]
        for i in range(rows):
            g = rng(cfg.seed, "shuffle", step, b, i)
            out[b * rows + i, :len(s)] = g.permutation(s)
    return out


def planted_logits(cfg: Config, device="cpu", p_plant: float = 0.7):
    """Logits [B][d+1][V] ~ N(0, 1) and drafts [B][d]. For each draft slot
    ``i < d``, with probability ``p_plant`` a uniformly drawn token gets the
    unique largest logit of row ``i`` (row max + 0.5); otherwise the draft is a
    uniform token whose logit is below the row max."""
    B, d, V = cfg.B, cfg.d, cfg.V
    dt = torch.float32 if cfg.logits_dtype == "f32" else torch.bfloat16
    g = torch.Generator(device=device)
    g.manual_seed(torch_seed(cfg.seed, "logits"))
    logits = torch.randn((B, d + 1, V), generator=g, device=device,
                         dtype=torch.float32).to(dt)
    drafts = np.zeros((B, d), dtype=np.int32)
    planted = np.zeros((B, d), dtype=bool)
    rowmax = logits[:, :d, :].float().amax(dim=2).cpu().numpy()
    for b in range(B):
        gb = rng(cfg.seed, "drafts", b)
        for i in range(d):
            if gb.random() < p_plant:
                tok = int(gb.integers(0, V))
                logits[b, i, tok] = float(rowmax[b, i]) + 0.5
                planted[b, i] = True
            else:
                row = logits[b, i].float().cpu().numpy()
                while True:
                    tok = int(gb.integers(0, V))
                    if row[tok] < rowmax[b, i]:
                        break
            drafts[b, i] = tok
    return logits, drafts, planted


# ------------------------------------------------------------ placement --
# Tensors of a workload on a device. These helpers only draw and place
# inputs; the path's arithmetic lives in the library and in the oracle.

def _i32(x, device):
    return torch.as_tensor(np.ascontiguousarray(x), dtype=torch.int32).to(device)


def blocks_needed(n_positions: int, block_size: int) -> int:
    return (int(n_positions) + block_size - 1) // block_size


def resident_case(cfg: Config, step: int = 0, device="cuda") -> dict:
    """Fully-resident workload: a paged latent cache covering every request's
    positions 0 .. L_b + d (a shuffled physical block table), q, and top-k."""
    req, ri = rows_of(cfg)
    clen = causal_lengths(cfg.L, req, ri)
    nblk = [blocks_needed(L + cfg.d + 1, cfg.block_size) for L in cfg.L]
    bt, total = shuffled_block_table(cfg.seed, "bt", nblk)
    kv = bf16_normal((total * cfg.block_size, LATENT), KV_SCALE, cfg.seed, "kvcache",
                     device=device)
    q = bf16_normal((cfg.R, cfg.H, LATENT), KV_SCALE, cfg.seed, "q", step, device=device)
    topk = topk_independent(cfg, step, cfg.L, req, ri)
    return dict(req=_i32(req, device), clen=_i32(clen, device), bt=_i32(bt, device),
                topk=_i32(topk, device), q=q, kv=kv, topk_np=topk, req_np=req,
                clen_np=clen, bt_np=bt)


def host_pool_tensor(rows: int, seed: int, device="cuda", pin=True) -> torch.Tensor:
    """A [rows][576] bf16 pool ~ N(0,1)/24 in page-locked host memory (drawn on
    ``device`` in chunks and copied down)."""
    pool = torch.empty((rows, LATENT), dtype=torch.bfloat16, pin_memory=pin)
    chunk = 1 << 19
    for c, start in enumerate(range(0, rows, chunk)):
        stop = min(rows, start + chunk)
        part = bf16_normal((stop - start, LATENT), KV_SCALE, seed, "hostpool", c,
                           device=device, chunk_rows=chunk)
        pool[start:stop].copy_(part)
    return pool


def host_backed_case(cfg: Config, device="cuda", extra_positions: int = 0) -> dict:
    """Host-backed workload: a paged page-locked host pool covering each
    request's positions 0 .. max_ctx - 1 (a shuffled host block table), an
    empty device hot buffer of B * (S + d + 1) rows, and kv_len = L."""
    bs = cfg.block_size
    max_ctx = max(cfg.L) + (cfg.d + 1) + extra_positions
    nblk = [blocks_needed(min(max_ctx, L + cfg.d + 1 + extra_positions), bs) for L in cfg.L]
    hbt, total = shuffled_block_table(cfg.seed, "hbt", nblk)
    width = blocks_needed(max_ctx, bs)
    if hbt.shape[1] < width:
        hbt = np.concatenate([hbt, np.full((cfg.B, width - hbt.shape[1]), -1, np.int32)], 1)
    pool = host_pool_tensor(total * bs, cfg.seed, device=device,
                            pin=torch.cuda.is_available())
    S_tot = cfg.S + cfg.d + 1
    hot = torch.zeros((cfg.B * S_tot, LATENT), dtype=torch.bfloat16, device=device)
    return dict(max_ctx=max_ctx, hbt=_i32(hbt, device), hbt_np=hbt, pool=pool, hot=hot,
                kv_len=_i32(np.asarray(cfg.L), device), S_tot=S_tot)


def step_kv(cfg: Config, step: int, device="cuda") -> torch.Tensor:
    """Fresh KV of each request's step positions L .. L + d (anchor + drafts)."""
    return bf16_normal((cfg.B, cfg.d + 1, LATENT), KV_SCALE, cfg.seed, "stepkv", step,
                       device=device)


def step_q(cfg: Config, step: int, device="cuda") -> torch.Tensor:
    return bf16_normal((cfg.R, cfg.H, LATENT), KV_SCALE, cfg.seed, "q", step, device=device)
