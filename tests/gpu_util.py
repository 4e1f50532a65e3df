"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

ABS_TOL = 1e-2      # max |gpu - oracle| over every output element
REL_TOL = 2e-2      # max |gpu - oracle| / max |oracle| per (row, head) vector


def lib():
    import __graft_entry__ as G
    G.build()
    import hisparse_top_sparse_gb300 as hs
    hs.lib()
    return hs


def np_(t):
    return t.detach().cpu().numpy()


def check_attn(out, ref, lse=None, ref_lse=None, rows=None):
    """out: GPU bf16 [R][H][512] (or a subset given by rows); ref float64."""
    x = out.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        x = x[rows]
    assert x.shape == ref.shape
    err = np.abs(x - ref)
    assert err.max() <= ABS_TOL, f"max abs error {err.max()}"
    denom = np.abs(ref).max(axis=-1)
    vec_err = err.max(axis=-1)
    zero = denom == 0
    assert np.all(vec_err[zero] == 0), "rows with no valid entry must be exactly 0"
    if (~zero).any():
        rel = vec_err[~zero] / denom[~zero]
        assert rel.max() <= REL_TOL, f"max per-vector relative error {rel.max()}"
    if lse is not None:
        y = lse.cpu().numpy().astype(np.float64)
        if rows is not None:
            y = y[rows]
        inf = np.isneginf(ref_lse)
        assert np.array_equal(np.isneginf(y), inf)
        d = np.abs(y[~inf] - ref_lse[~inf])
        if d.size:
            assert (d <= 1e-4 + 1e-5 * np.abs(ref_lse[~inf])).all(), f"lse error {d.max()}"
    return err.max()
